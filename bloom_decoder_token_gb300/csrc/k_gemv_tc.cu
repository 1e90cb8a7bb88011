// Decode linear layers on the 5th-generation tensor cores (tcgen05 + TMEM + TMA), sm_103a.
//
// y[m][n] = epilogue(sum_k x[m][k] W[n][k]) for the B tokens of a decode step
// (B up to 256).  At decode the time is the time to stream W once ("DeepSpeed
// Inference", III.A); the weight-streaming mma.sync kernel does that well for
// one or two tokens, but from 8 tokens on its registers and shared-memory
// traffic per weight byte grow with B.  Here W is the MMA's A operand (128
// weight rows per tile) and the step's tokens are its N operand (NT = B rounded
// up to 16, 32, 64, 128 or 256 columns), so the tensor cores take any batch at
// no extra cost per weight byte:
//  * warp 0, one lane: TMA producer.  Each stage holds a 128 x 64 weight tile
//    and the NT x 64 activation tile of the same k (2-D tensor maps, 128-byte
//    swizzle).  The weight tiles of the first stages are requested before the
//    kernel waits for its predecessor (programmatic dependent launch); the
//    activations, which that kernel writes, after;
//  * warp 1, one lane: tcgen05.mma kind::f16 (M = 128, N = NT, K = 16, four per
//    stage) accumulating in TMEM; tcgen05.commit frees each stage;
//  * warps 2-5: epilogue, one TMEM lane (= weight row) per thread, 16 token
//    columns per tcgen05.ld: bias, GeLU, float32 residual add, the Q/K/V
//    scatter into the cache slot of the step, or the LM head's logits and
//    argmax (the fusions of "DeepSpeed Inference", III.D).
// In the decode step this kernel runs the tied LM head (the largest single
// weight stream: V x h) for 8 or more sequences, where it streams at twice the
// weight-streaming kernel's rate (2 GB head of the 7b1 shape, 32 sequences:
// 334 us vs 675 us), and the bf16 block linears from 8 sequences on where
// they are wide or long (7b1 shape, 32 sequences: up 26 us vs 49 us).
// Narrow matrices split K over several CTAs so that the grid fills the GPU;
// each split stores its float32 partial tile and the last split of a row tile
// to finish (a ticket, no waiting) sums the partials in split order, so the
// result does not depend on timing.  Every mbarrier wait is bounded (about two
// seconds of SM clock); on expiry the kernel records kErrTimeout, skips its
// stores and still frees TMEM.
#include "common.cuh"
#include "kernels.h"
#include "tc_ops.cuh"
#include "tile_ops.cuh"

namespace bloom {

constexpr int kGvRows = 128;                      // weight rows per tile (MMA M)
constexpr int kGvBK = 64;                         // k per stage: one 128-byte swizzle row
constexpr int kGvThreads = 192;                   // 6 warps
constexpr int kGvWBytes = kGvRows * kGvBK * 2;    // 16 KB
constexpr int kGvSmemBudget = 108 * 1024;         // two CTAs per SM
constexpr int kGvTargetCtas = 120;                // CTAs a K split aims for

template <int NT>
struct GvCfg {
    static constexpr int XBytes = NT * kGvBK * 2;
    static constexpr int Stage = kGvWBytes + XBytes;
    static constexpr int StagesFit = kGvSmemBudget / Stage;
    static constexpr int Stages = StagesFit > 8 ? 8 : (StagesFit < 2 ? 2 : StagesFit);
    static constexpr size_t Smem = (size_t)Stages * Stage + 1024;   // + alignment slack
    static constexpr int TmemCols = NT < 32 ? 32 : NT;
};

__device__ __forceinline__ void epi_bar_sync() {   // the four epilogue warps only
    asm volatile("bar.sync 1, 128;" ::: "memory");
}

// Epilogue of one (row n, token m) value.
template <int EPI>
__device__ __forceinline__ void gv_apply(const LinearArgs &a, int m, int n, float v, float bias,
                                         int slot, unsigned long long &best) {
    v += bias;
    const size_t o = (size_t)m * a.N + n;
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
        const int hj = n / (3 * dh);
        const int cidx = (n / dh) % 3;
        const int e = n % dh;
        if (cidx == 0) {
            a.q_out[(size_t)m * a.n_head * dh + (size_t)hj * dh + e] = f2bf(v);
        } else if (slot >= 0 && slot < a.max_seq) {
            uint16_t *cache = (cidx == 1) ? a.k_cache : a.v_cache;
            cache[(((size_t)m * a.n_head + hj) * a.max_seq + slot) * dh + e] = f2bf(v);
        } else if (a.err) {
            atomicOr(a.err, kErrSlot);
        }
    } else if constexpr (EPI == EPI_ARGMAX) {
        if (a.logits) a.logits[o] = v;
        best = pack_argmax(v, (uint32_t)n);
    }
}

template <int EPI, int NT>
__global__ void __launch_bounds__(kGvThreads, 1)
gemv_tc_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
               const GemvTcArgs g) {
    using C = GvCfg<NT>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        ((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    __shared__ uint64_t full[C::Stages], empty[C::Stages], acc_full;
    __shared__ uint32_t tmem_base;
    __shared__ int s_abort, s_last_tile, s_last;
    __shared__ unsigned long long s_best[EPI == EPI_ARGMAX ? kMaxBatch : 1];

    const LinearArgs &a = g.a;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tile = blockIdx.x, split = blockIdx.y;
    const int n0 = tile * kGvRows;
    const int nkb = (a.K + kGvBK - 1) / kGvBK;
    const int per = (nkb + g.splits - 1) / g.splits;
    const int kb0 = split * per;
    const int kb1 = min(nkb, kb0 + per);
    const int my_kb = kb1 > kb0 ? kb1 - kb0 : 0;

    if (tid == 0) {
        for (int s = 0; s < C::Stages; ++s) {
            tc_mbar_init(&full[s], 1);
            tc_mbar_init(&empty[s], 1);
        }
        tc_mbar_init(&acc_full, 1);
        s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tm_w) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tm_x) : "memory");
    }
    if constexpr (EPI == EPI_ARGMAX) {
        for (int i = tid; i < NT; i += blockDim.x) s_best[i] = 0ull;
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         tc_smem(&tmem_base)),
                     "n"(C::TmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = tmem_base;
    griddep_launch();

    if (warp == 0) {
        if (lane == 0) {
            // ---- TMA producer.  Weight tiles of the first stages go out before the
            // wait for the previous kernel (they do not depend on it).
            const int pre = my_kb < C::Stages ? my_kb : C::Stages;
            for (int i = 0; i < pre; ++i) {
                unsigned char *st = smem + (size_t)i * C::Stage;
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
                                 tc_smem(&full[i])),
                             "r"(C::Stage)
                             : "memory");
                tc_tma_2d(st, &tm_w, (kb0 + i) * kGvBK, n0, &full[i]);
            }
            griddep_wait();   // the activations come from the previous kernel
            for (int i = 0; i < pre; ++i)
                tc_tma_2d(smem + (size_t)i * C::Stage + kGvWBytes, &tm_x, (kb0 + i) * kGvBK, 0,
                          &full[i]);
            int issued = pre;
            for (int i = pre; i < my_kb; ++i) {
                const int s = i % C::Stages;
                if (!tc_mbar_wait(&empty[s], (uint32_t)(((i / C::Stages) & 1) ^ 1))) {
                    s_abort = 1;
                    if (a.err) atomicOr(a.err, kErrTimeout);
                    break;
                }
                unsigned char *st = smem + (size_t)s * C::Stage;
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
                                 tc_smem(&full[s])),
                             "r"(C::Stage)
                             : "memory");
                tc_tma_2d(st, &tm_w, (kb0 + i) * kGvBK, n0, &full[s]);
                tc_tma_2d(st + kGvWBytes, &tm_x, (kb0 + i) * kGvBK, 0, &full[s]);
                ++issued;
            }
            // no copy of ours may still be landing when the CTA exits
            for (int j = 0; j < C::Stages && j < issued; ++j) {
                const int i = issued - 1 - j;
                if (!tc_mbar_wait(&full[i % C::Stages], (uint32_t)((i / C::Stages) & 1)) && a.err)
                    atomicOr(a.err, kErrTimeout);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---- MMA issuer
            constexpr uint32_t idesc = tc_idesc(kGvRows, NT);
            bool ok = true;
            for (int i = 0; i < my_kb; ++i) {
                const int s = i % C::Stages;
                if (!tc_mbar_wait(&full[s], (uint32_t)((i / C::Stages) & 1))) {
                    ok = false;
                    break;
                }
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t sw = tc_smem(smem + (size_t)s * C::Stage);
                const uint64_t dw = tc_desc(sw), dx = tc_desc(sw + kGvWBytes);
#pragma unroll
                for (int k = 0; k < kGvBK / 16; ++k)   // 16 bf16 = 32 bytes per step
                    tc_mma(tmem, dw + (uint64_t)(2 * k), dx + (uint64_t)(2 * k), idesc,
                           (i > 0 || k > 0) ? 1u : 0u);
                tc_commit(&empty[s]);
            }
            if (!ok) {
                s_abort = 1;
                if (a.err) atomicOr(a.err, kErrTimeout);
            }
            tc_commit(&acc_full);   // accumulator complete (or abandoned)
        }
    } else {
        // ---- epilogue: warps 2..5 -> TMEM lane quarters (warp % 4); thread = weight row
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const int n = n0 + r;
        const bool nok = n < a.N;
        griddep_wait();   // the residual and the cache belong to earlier kernels too
        const float bias = (a.bias && nok) ? bf2f(a.bias[n]) : 0.f;
        const int slot = (EPI == EPI_QKV && a.len_ptr) ? *a.len_ptr : 0;
        // longer limit than the MMA issuer's, so that its final commit arrives first
        const bool ok = tc_mbar_wait(&acc_full, 0, 3 * kTcWaitCycles);
        if (!ok && a.err) atomicOr(a.err, kErrTimeout);
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        // warp-uniform, so that the argmax shuffles below see every lane
        const bool live = __all_sync(0xffffffffu, ok && !*(volatile int *)&s_abort);
        const int mmax = a.M < NT ? a.M : NT;
        const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16);
        if (g.splits == 1) {
#pragma unroll 1
            for (int c = 0; c < NT; c += 16) {
                float v[16];
                tc_ld16(taddr + (uint32_t)c, v);   // whole warp
                if (!live) continue;               // warp-uniform
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int m = c + j;
                    if (m >= mmax) break;          // warp-uniform
                    unsigned long long best = 0;   // rows past N take no part
                    if (nok) gv_apply<EPI>(a, m, n, my_kb ? v[j] : 0.f, bias, slot, best);
                    if constexpr (EPI == EPI_ARGMAX) {
                        // max over the warp's 32 rows (every lane shuffles), then the CTA's
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) {
                            const unsigned long long ob = __shfl_xor_sync(0xffffffffu, best, o);
                            best = ob > best ? ob : best;
                        }
                        if (lane == 0 && best) atomicMax(&s_best[m], best);
                    }
                }
            }
        } else {
            // split K: store this split's partial tile [NT][128], the last split sums
            float *mine = g.part + ((size_t)tile * g.splits + split) * NT * kGvRows;
#pragma unroll 1
            for (int c = 0; c < NT; c += 16) {
                float v[16];
                tc_ld16(taddr + (uint32_t)c, v);
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (c + j < mmax) mine[(size_t)(c + j) * kGvRows + r] = (live && my_kb) ? v[j] : 0.f;
            }
            __threadfence();
            epi_bar_sync();
            if (tid == 64) s_last_tile = (atomicAdd(g.ticket + tile, 1) == g.splits - 1);
            epi_bar_sync();
            if (s_last_tile) {
                __threadfence();
                const float *base = g.part + (size_t)tile * g.splits * NT * kGvRows;
                for (int m = 0; m < mmax; ++m) {
                    float t = 0.f;
                    for (int sp = 0; sp < g.splits; ++sp)
                        t += __ldcg(base + ((size_t)sp * NT + m) * kGvRows + r);
                    unsigned long long best = 0;
                    if (live && nok) gv_apply<EPI>(a, m, n, t, bias, slot, best);
                }
                if (tid == 64) g.ticket[tile] = 0;
            }
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "n"(C::TmemCols));
    }
    if constexpr (EPI == EPI_ARGMAX) argmax_publish(a, s_best, &s_last, tid, gridDim.x * gridDim.y);
}

// ---------------------------------------------------------------- host side
int gemv_tc_nt(int M) {
    if (M <= 16) return 16;
    if (M <= 32) return 32;
    if (M <= 64) return 64;
    if (M <= 128) return 128;
    return M <= 256 ? 256 : 0;
}

// K splits per row tile: the fewest that fill the GPU's CTA slots (two CTAs
// per SM) in whole waves, at most one split per 4 k-blocks.
// K splits of a launch: enough CTAs for about kGvTargetCtas SMs and no more.
// Measured on GB300 at 16-64 tokens, an unsplit 96- or 128-tile matrix streams
// at 65-79 % of the copy peak while 2-7 splits of it (more CTAs, each partial
// tile written, and summed by the last split) ran at 27-55 %; a 32-tile matrix
// wants 4.
int gemv_tc_splits(int N, int K, int num_sms, int epi) {
    (void)num_sms;
    if (epi == EPI_ARGMAX) return 1;
    const int tiles = (N + kGvRows - 1) / kGvRows;
    const int nkb = (K + kGvBK - 1) / kGvBK;
    int s = (kGvTargetCtas + tiles / 2) / tiles;   // rounded: 96 or 128 tiles -> 1, 32 -> 4
    if (s > 16) s = 16;
    while (s > 1 && s * 4 > nkb) --s;   // at least 4 k-blocks per split
    return s < 1 ? 1 : s;
}

size_t gemv_tc_part_floats(int N, int K, int M, int num_sms) {
    const int nt = gemv_tc_nt(M);
    const int tiles = (N + kGvRows - 1) / kGvRows;
    const int s = gemv_tc_splits(N, K, num_sms, EPI_STORE);
    return s > 1 ? (size_t)tiles * s * nt * kGvRows : 0;
}

int gemv_tc_box_rows_w() { return kGvRows; }

template <int EPI, int NT>
static cudaError_t gv_launch_t(const void *mw, const void *mx, const GemvTcArgs &g, cudaStream_t s) {
    using C = GvCfg<NT>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(gemv_tc_kernel<EPI, NT>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::Smem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const CUtensorMap &tw = *reinterpret_cast<const CUtensorMap *>(mw);
    const CUtensorMap &tx = *reinterpret_cast<const CUtensorMap *>(mx);
    dim3 grid((g.a.N + kGvRows - 1) / kGvRows, g.splits);
    return launch_pdl_smem(gemv_tc_kernel<EPI, NT>, grid, dim3(kGvThreads), C::Smem, s, tw, tx, g);
}

template <int EPI>
static cudaError_t gv_launch_epi(const void *mw, const void *mx, const GemvTcArgs &g, int nt,
                                 cudaStream_t s) {
    switch (nt) {
        case 16: return gv_launch_t<EPI, 16>(mw, mx, g, s);
        case 32: return gv_launch_t<EPI, 32>(mw, mx, g, s);
        case 64: return gv_launch_t<EPI, 64>(mw, mx, g, s);
        case 128: return gv_launch_t<EPI, 128>(mw, mx, g, s);
        case 256: return gv_launch_t<EPI, 256>(mw, mx, g, s);
        default: return cudaErrorInvalidValue;
    }
}

template <int EPI>
static cudaError_t gv_prepare_epi() {
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(gemv_tc_kernel<EPI, 16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)GvCfg<16>::Smem)))
        return e;
    if ((e = cudaFuncSetAttribute(gemv_tc_kernel<EPI, 32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)GvCfg<32>::Smem)))
        return e;
    if ((e = cudaFuncSetAttribute(gemv_tc_kernel<EPI, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)GvCfg<64>::Smem)))
        return e;
    if ((e = cudaFuncSetAttribute(gemv_tc_kernel<EPI, 128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)GvCfg<128>::Smem)))
        return e;
    return cudaFuncSetAttribute(gemv_tc_kernel<EPI, 256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)GvCfg<256>::Smem);
}

cudaError_t gemv_tc_prepare() {
    cudaError_t e;
    if ((e = gv_prepare_epi<EPI_STORE>())) return e;
    if ((e = gv_prepare_epi<EPI_GELU>())) return e;
    if ((e = gv_prepare_epi<EPI_RESID>())) return e;
    if ((e = gv_prepare_epi<EPI_RESID32>())) return e;
    if ((e = gv_prepare_epi<EPI_QKV>())) return e;
    return gv_prepare_epi<EPI_ARGMAX>();
}

cudaError_t launch_gemv_tc(const void *map_w, const void *map_x, const GemvTcArgs &g, int nt,
                           cudaStream_t s) {
    const LinearArgs &a = g.a;
    if (a.M <= 0 || a.N <= 0) return cudaSuccess;
    if (a.int8 || a.K % 8 || a.T != 0 || gemv_tc_nt(a.M) != nt || a.M > kMaxBatch) return cudaErrorInvalidValue;
    if (g.splits < 1 || (g.splits > 1 && (!g.part || !g.ticket || a.epi == EPI_ARGMAX)))
        return cudaErrorInvalidValue;
    switch (a.epi) {
        case EPI_STORE: return gv_launch_epi<EPI_STORE>(map_w, map_x, g, nt, s);
        case EPI_GELU: return gv_launch_epi<EPI_GELU>(map_w, map_x, g, nt, s);
        case EPI_RESID: return gv_launch_epi<EPI_RESID>(map_w, map_x, g, nt, s);
        case EPI_RESID32: return gv_launch_epi<EPI_RESID32>(map_w, map_x, g, nt, s);
        case EPI_QKV: return gv_launch_epi<EPI_QKV>(map_w, map_x, g, nt, s);
        case EPI_ARGMAX: return gv_launch_epi<EPI_ARGMAX>(map_w, map_x, g, nt, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace bloom
