// Decode linear layers on the 5th-generation tensor cores (tcgen05 + TMEM + TMA), sm_103a.
//
// y[m][n] = epilogue(sum_k x[m][k] W[n][k]) for the B tokens of a decode step
// (B up to 256).  At decode the time is the time to stream W once ("DeepSpeed
// Inference", III.A).  W is the MMA's A operand (128 weight rows per tile)
// and the step's tokens are its N operand (NT = B rounded up to 16, 32, 64,
// 128 or 256 columns), so the tensor cores take any batch at no extra cost
// per weight byte:
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
//
// The grid is (row tiles) x (K splits), two CTAs per SM (about 100 KB of
// weights in flight each).  A matrix with few row tiles (4096 rows = 32 tiles)
// would leave most SMs idle, so K is split S ways (gemv_tc_splits).  The S
// splits of a row tile run as one thread-block cluster: each token group of 4
// is finished by one CTA of the cluster, every split pushes its float32
// partial of that group into the finisher's shared memory (distributed shared
// memory stores, no waiting on loads), and after a cluster barrier each CTA
// sums what it received in split order -- the result does not depend on
// timing, and no global scratch or second pass is needed (the cross-CTA
// reduction of SBI-GeMM, "DeepSpeed Inference", III.C.2, kept on chip).  The
// residuals a finisher adds are loaded during the main loop.
//
// Every mbarrier wait is bounded (about two seconds of SM clock); on expiry
// the kernel records kErrTimeout, skips its stores and still frees TMEM.  The
// two cluster barriers are reached on every path (every wait before them is
// bounded), so no CTA of a cluster waits on a peer that has left, and no CTA
// writes into a peer's shared memory after that peer has passed the second.
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
constexpr int kGvMaxSplits = 16;                  // largest cluster (non-portable size)
constexpr int kGvMinKbPerSplit = 4;               // k-blocks a split streams at least

// W8: int8 weights.  A stage then holds a 128 x 128 int8 weight tile (the same
// 16 KB) and the NT x 128 activations (two 64-wide boxes); the epilogue warps
// widen each stage's codes into one of two TMEM A buffers (64 columns of 16-bit
// pairs each, columns [0, 128)), the accumulator sits at column 128.  Up to 32
// token columns the codes are widened to f16 (two instructions a pair) and the
// stage's activations converted to f16 in place, so that the MMA (kind::f16)
// takes f16 A and B; above, where converting the activations costs more than
// it saves, to bf16 (four a pair) with the activations as they are.  Measured
// on GB300 (7b1 int8, decode step): 8 sequences 2.479 ms with f16 vs 2.610
// bf16, 32: 2.945 vs 2.974, 128: 6.015 vs 5.557.
template <int NT, bool W8>
constexpr bool kGvW8F16 = W8 && NT <= 32;
template <bool F16>
__device__ __forceinline__ uint32_t gv_widen(uint32_t w, int i) {
    if constexpr (F16) return i8x2_to_f16x2(w, i);
    else return i8x2_to_bf16x2(w, i);
}
template <int NT, bool W8 = false>
struct GvCfg {
    static constexpr int KB = W8 ? 128 : kGvBK;   // k per stage
    static constexpr int XBytes = NT * KB * 2;
    static constexpr int Stage = kGvWBytes + XBytes;
    static constexpr int StagesFit = kGvSmemBudget / Stage;
    static constexpr int Stages = StagesFit > 8 ? 8 : (StagesFit < 2 ? 2 : StagesFit);
    static constexpr size_t Smem = (size_t)Stages * Stage + 1024;   // + alignment slack
    static constexpr int TmemCols = W8 ? 256 : (NT < 32 ? 32 : NT);
    static constexpr uint32_t AccCol = W8 ? 128u : 0u;
    // K split: the receive area of pushed partials, [split][128 rows][groups
    // this CTA finishes] float4 (4 tokens), lives in the idle ring; at most
    // NT / 4 + kGvMaxSplits float4 per row
    static constexpr bool CanSplit =
        (size_t)(NT / 4 + kGvMaxSplits) * kGvRows * 16 <= (size_t)Stages * Stage;
};

// ---- cluster helpers (distributed shared memory)
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t dsmem_map(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}
__device__ __forceinline__ void st_dsmem4(uint32_t addr, float4 v) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "f"(v.x), "f"(v.y),
                 "f"(v.z), "f"(v.w)
                 : "memory");
}

// The cache slot a decode token's K and V go to (staged per CTA in shared
// memory), or kGvNoSlot for an idle row.
constexpr int kGvNoSlot = -0x40000000;

// Epilogue of J consecutive tokens m0.. of one row n (v: accumulators, the
// bias not yet added).  The residual epilogues take the residual values in
// `res` when the caller loaded them ahead (during the main loop), else every
// load is issued before any store, so the J tokens cost one memory round trip.
template <int EPI, int J>
__device__ __forceinline__ void gv_apply(const LinearArgs &a, int m0, int mmax, int n, const float *v,
                                         float bias, const int *slots, unsigned long long *best,
                                         const float *res = nullptr) {
    if constexpr (EPI == EPI_RESID32 || EPI == EPI_RESID) {
        float r[J];
#pragma unroll
        for (int j = 0; j < J; ++j) {
            if (res) {
                r[j] = res[j];
            } else if (m0 + j < mmax) {
                if constexpr (EPI == EPI_RESID32) r[j] = a.out32[(size_t)(m0 + j) * a.N + n];
                else r[j] = bf2f(a.out[(size_t)(m0 + j) * a.N + n]);
            } else {
                r[j] = 0.f;
            }
        }
#pragma unroll
        for (int j = 0; j < J; ++j) {
            if (m0 + j >= mmax) break;
            if constexpr (EPI == EPI_RESID32) a.out32[(size_t)(m0 + j) * a.N + n] = r[j] + (v[j] + bias);
            else a.out[(size_t)(m0 + j) * a.N + n] = f2bf(r[j] + (v[j] + bias));
        }
    } else {
#pragma unroll
        for (int j = 0; j < J; ++j) {
            const int m = m0 + j;
            if (m >= mmax) break;
            const float x = v[j] + bias;
            const size_t o = (size_t)m * a.N + n;
            if constexpr (EPI == EPI_STORE) {
                a.out[o] = f2bf(x);
            } else if constexpr (EPI == EPI_GELU) {
                a.out[o] = f2bf(gelu_tanh(x));
            } else if constexpr (EPI == EPI_QKV) {
                const int dh = a.head_dim;
                const int hj = n / (3 * dh);
                const int cidx = (n / dh) % 3;
                const int e = n % dh;
                if (cidx == 0) {
                    a.q_out[(size_t)m * a.n_head * dh + (size_t)hj * dh + e] = f2bf(x);
                } else if (slots[m] != kGvNoSlot) {   // an idle row appends nothing
                    const int slot = slots[m];
                    if (slot >= 0 && slot < a.max_seq) {
                        uint16_t *cache = (cidx == 1) ? a.k_cache : a.v_cache;
                        cache[(((size_t)m * a.n_head + hj) * a.max_seq + slot) * dh + e] = f2bf(x);
                    } else if (a.err) {
                        atomicOr(a.err, kErrSlot);
                    }
                }
            } else if constexpr (EPI == EPI_ARGMAX) {
                if (a.logits) a.logits[o] = x;
                best[j] = pack_argmax(x, (uint32_t)n);
            }
        }
    }
}

// Token groups (4 tokens) whose residuals a CTA of a K split loads ahead.
constexpr int kGvResGroups = 4;

template <int EPI, int NT, bool W8>
__global__ void __launch_bounds__(kGvThreads, 1)
gemv_tc_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
               const GemvTcArgs g) {
    using C = GvCfg<NT, W8>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        ((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    __shared__ uint64_t full[C::Stages], empty[C::Stages], acc_full;
    __shared__ uint64_t a_full[W8 ? 2 : 1], a_empty[W8 ? 2 : 1];   // TMEM A buffers (W8)
    __shared__ uint32_t tmem_base;
    __shared__ int s_abort, s_last;
    __shared__ unsigned long long s_best[EPI == EPI_ARGMAX ? kMaxBatch : 1];
    __shared__ int s_slot[EPI == EPI_QKV ? NT : 1];

    const LinearArgs &a = g.a;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tile = blockIdx.x, split = blockIdx.y;   // the cluster spans the splits
    const int n0 = tile * kGvRows;
    const int nkb = (a.K + C::KB - 1) / C::KB;
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
        if constexpr (W8) {
            for (int b = 0; b < 2; ++b) {
                tc_mbar_init(&a_full[b], 4);    // one arrival per converting warp
                tc_mbar_init(&a_empty[b], 1);   // the MMA issuer's commit
            }
        }
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
            auto load_x = [&](unsigned char *st, int i, uint64_t *bar) {
#pragma unroll
                for (int h = 0; h < C::KB / kGvBK; ++h)
                    tc_tma_2d(st + kGvWBytes + h * NT * 128, &tm_x, (kb0 + i) * C::KB + h * kGvBK, 0,
                              bar);
            };
            const int pre = my_kb < C::Stages ? my_kb : C::Stages;
            for (int i = 0; i < pre; ++i) {
                unsigned char *st = smem + (size_t)i * C::Stage;
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
                                 tc_smem(&full[i])),
                             "r"(C::Stage)
                             : "memory");
                tc_tma_2d(st, &tm_w, (kb0 + i) * C::KB, n0, &full[i]);
            }
            griddep_wait();   // the activations come from the previous kernel
            for (int i = 0; i < pre; ++i) load_x(smem + (size_t)i * C::Stage, i, &full[i]);
            int issued = pre;
            for (int i = pre; i < my_kb; ++i) {
                const int s = i % C::Stages;
                if (!tc_mbar_wait(&empty[s], (uint32_t)(((i / C::Stages) & 1) ^ 1), a.wait_ns)) {
                    s_abort = 1;
                    if (a.err) atomicOr(a.err, kErrTimeout);
                    break;
                }
                unsigned char *st = smem + (size_t)s * C::Stage;
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
                                 tc_smem(&full[s])),
                             "r"(C::Stage)
                             : "memory");
                tc_tma_2d(st, &tm_w, (kb0 + i) * C::KB, n0, &full[s]);
                load_x(st, i, &full[s]);
                ++issued;
            }
            // no copy of ours may still be landing when the stages are reused or
            // the CTA exits
            for (int j = 0; j < C::Stages && j < issued; ++j) {
                const int i = issued - 1 - j;
                if (!tc_mbar_wait(&full[i % C::Stages], (uint32_t)((i / C::Stages) & 1), kTcWaitNs) &&
                    a.err)
                    atomicOr(a.err, kErrTimeout);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---- MMA issuer
            // int8 up to 32 columns: both operands f16 (the widened codes and the
            // converted activations); otherwise both bf16
            constexpr uint32_t idesc = tc_idesc(kGvRows, NT, kGvW8F16<NT, W8>);
            const uint32_t acc = tmem + C::AccCol;
            bool ok = true;
            for (int i = 0; i < my_kb; ++i) {
                const int s = i % C::Stages;
                if (!tc_mbar_wait(&full[s], (uint32_t)((i / C::Stages) & 1), a.wait_ns)) {
                    ok = false;
                    break;
                }
                const uint32_t sw = tc_smem(smem + (size_t)s * C::Stage);
                if constexpr (W8) {
                    // the widened weights of this stage, in TMEM A buffer i % 2
                    if (!tc_mbar_wait(&a_full[i & 1], (uint32_t)((i >> 1) & 1), a.wait_ns)) {
                        ok = false;
                        break;
                    }
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    const uint32_t ta = tmem + (uint32_t)((i & 1) * 64);
#pragma unroll
                    for (int k = 0; k < C::KB / 16; ++k) {   // 8 steps of 16: two activation boxes
                        const uint64_t dx = tc_desc(sw + kGvWBytes + (k / 4) * NT * 128) + (uint64_t)(2 * (k % 4));
                        tc_mma_tmem_a(acc, ta + (uint32_t)(8 * k), dx, idesc, (i > 0 || k > 0) ? 1u : 0u);
                    }
                    tc_commit(&empty[s]);
                    tc_commit(&a_empty[i & 1]);
                } else {
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    const uint64_t dw = tc_desc(sw), dx = tc_desc(sw + kGvWBytes);
#pragma unroll
                    for (int k = 0; k < kGvBK / 16; ++k)   // 16 bf16 = 32 bytes per step
                        tc_mma(acc, dw + (uint64_t)(2 * k), dx + (uint64_t)(2 * k), idesc,
                               (i > 0 || k > 0) ? 1u : 0u);
                    tc_commit(&empty[s]);
                }
            }
            if (!ok) {
                s_abort = 1;
                if (a.err) atomicOr(a.err, kErrTimeout);
            }
            tc_commit(&acc_full);   // accumulator complete (or abandoned)
            // every MMA of ours has finished before TMEM is read or freed, on every path
            if (!tc_mbar_wait(&acc_full, 0, kTcWaitNs) && a.err) atomicOr(a.err, kErrTimeout);
        }
    }
    __syncwarp();

    // ---- epilogue: warps 2..5 -> TMEM lane quarters (warp % 4); thread = weight row
    const bool epi_warp = warp >= 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int n = n0 + r;
    const bool nok = n < a.N;
    const int mmax = a.M < NT ? a.M : NT;
    const int S = g.splits;
    const int groups = (mmax + 3) / 4;
    float bias = 0.f;
    bool live = false;
    // residuals of the token groups this CTA finishes (split, split + S, ...),
    // loaded while the main loop runs
    constexpr bool kRes = (EPI == EPI_RESID32 || EPI == EPI_RESID) && C::CanSplit;
    float res[kRes ? 4 * kGvResGroups : 1];
    const uint32_t tlane = tmem + ((uint32_t)(quarter * 32) << 16);
    float scale = 1.f;
    if (epi_warp) {
        if constexpr (W8) {
            // widen this thread's weight row of every stage (128 int8 codes, exact in
            // f16 and bf16) into TMEM A buffer i % 2 for the MMA issuer; in the f16
            // form also convert the stage's activations (one type for both operands)
            for (int i = 0; i < my_kb; ++i) {
                const int s = i % C::Stages;
                const bool wok = __all_sync(
                    0xffffffffu, tc_mbar_wait(&full[s], (uint32_t)((i / C::Stages) & 1), a.wait_ns) &&
                                     (i < 2 || tc_mbar_wait(&a_empty[i & 1], (uint32_t)(((i >> 1) - 1) & 1),
                                                            a.wait_ns)));
                if (!wok) {   // warp-uniform
                    s_abort = 1;
                    if (a.err) atomicOr(a.err, kErrTimeout);
                    break;
                }
                const unsigned char *wrow = smem + (size_t)s * C::Stage + (size_t)r * 128;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    uint32_t w[32];
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        const int c = hh * 4 + cc;   // 16-byte chunk, swizzled by the row
                        const uint4 q = *reinterpret_cast<const uint4 *>(wrow + ((c ^ (r & 7)) << 4));
                        w[cc * 8 + 0] = gv_widen<kGvW8F16<NT, W8>>(q.x, 0);
                        w[cc * 8 + 1] = gv_widen<kGvW8F16<NT, W8>>(q.x, 2);
                        w[cc * 8 + 2] = gv_widen<kGvW8F16<NT, W8>>(q.y, 0);
                        w[cc * 8 + 3] = gv_widen<kGvW8F16<NT, W8>>(q.y, 2);
                        w[cc * 8 + 4] = gv_widen<kGvW8F16<NT, W8>>(q.z, 0);
                        w[cc * 8 + 5] = gv_widen<kGvW8F16<NT, W8>>(q.z, 2);
                        w[cc * 8 + 6] = gv_widen<kGvW8F16<NT, W8>>(q.w, 0);
                        w[cc * 8 + 7] = gv_widen<kGvW8F16<NT, W8>>(q.w, 2);
                    }
                    tc_st32(tlane + (uint32_t)((i & 1) * 64 + hh * 32), w);
                }
                if constexpr (kGvW8F16<NT, W8>) {
                    // the stage's activations, bf16 -> f16 in place (NT x 128 values,
                    // 16 bytes a chunk), published to the tensor cores before the arrival
                    uint4 *xs = reinterpret_cast<uint4 *>(smem + (size_t)s * C::Stage + kGvWBytes);
                    for (int cx = tid - 64; cx < NT * 16; cx += 128) xs[cx] = bf16x8_to_f16x8(xs[cx]);
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                }
                tc_wait_st();
                asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
                __syncwarp();
                if (lane == 0)
                    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc_smem(&a_full[i & 1]))
                                 : "memory");
            }
            scale = nok ? bf2f(a.scale[n]) : 0.f;
        }
        griddep_wait();   // the residual and the cache belong to earlier kernels too
        bias = (a.bias && nok) ? bf2f(a.bias[n]) : 0.f;
        if constexpr (EPI == EPI_QKV) {
            const int ep = tid - 64;
            if (ep < NT)
                s_slot[ep] = (ep < a.M && (!a.active || a.active[ep])) ? a.len_ptr[ep] : kGvNoSlot;
            asm volatile("bar.sync 1, 128;" ::: "memory");   // the four epilogue warps
        }
        if constexpr (kRes) {
            if (S > 1) {
#pragma unroll
                for (int q = 0; q < kGvResGroups; ++q)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int m = (split + q * S) * 4 + j;
                        float v = 0.f;
                        if (nok && m < mmax) {
                            if constexpr (EPI == EPI_RESID32) v = a.out32[(size_t)m * a.N + n];
                            else v = bf2f(a.out[(size_t)m * a.N + n]);
                        }
                        res[4 * q + j] = v;
                    }
            }
        }
        // longer limit than the MMA issuer's, so that its final commit arrives first
        const bool ok = tc_mbar_wait(&acc_full, 0, 3 * (a.wait_ns ? a.wait_ns : kTcWaitNs));
        if (!ok && a.err) atomicOr(a.err, kErrTimeout);
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        // warp-uniform, so that the argmax shuffles below see every lane
        live = __all_sync(0xffffffffu, ok && !*(volatile int *)&s_abort);
    }
    const uint32_t taddr = tlane + C::AccCol;
    if (S == 1) {
        if (epi_warp) {
#pragma unroll 1
            for (int c = 0; c < NT; c += 16) {
                float v[16];
                tc_ld16(taddr + (uint32_t)c, v);   // whole warp
                if (!live || c >= mmax) continue;  // warp-uniform
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] = my_kb ? v[j] * scale : 0.f;
                unsigned long long best[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) best[j] = 0;   // rows past N take no part
                if (nok) gv_apply<EPI, 16>(a, c, mmax, n, v, bias, s_slot, best);
                if constexpr (EPI == EPI_ARGMAX) {
                    // max over the warp's 32 rows (every lane shuffles), then the CTA's
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        unsigned long long b = best[j];
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) {
                            const unsigned long long ob = __shfl_xor_sync(0xffffffffu, b, o);
                            b = ob > b ? ob : b;
                        }
                        if (lane == 0 && b && c + j < mmax) atomicMax(&s_best[c + j], b);
                    }
                }
            }
        }
    } else if constexpr (C::CanSplit && EPI != EPI_ARGMAX) {
        // K split over the cluster.  Token group gi (4 tokens) is finished by the
        // CTA of rank gi % S; every split pushes its partial of that group into
        // the finisher's receive area [split][128 rows][gpc] (float4), in the
        // finisher's ring, which is idle once every split is past its main loop
        // (all its MMAs have completed and every copy into it has landed).
        const int gpc = (groups + S - 1) / S;
        float4 *recv = reinterpret_cast<float4 *>(smem);
        __syncwarp();
        cluster_arrive();   // this CTA's ring is idle
        cluster_wait();     // ... and every peer's
        if (epi_warp) {
            const uint32_t rb = tc_smem(recv);
            const bool use = live && my_kb > 0;
#pragma unroll 1
            for (int c = 0; c < NT; c += 16) {
                float v[16];
                tc_ld16(taddr + (uint32_t)c, v);   // whole warp
                if (c >= mmax) continue;           // warp-uniform
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int gi = c / 4 + q;
                    if (gi >= groups) break;
                    const float4 val = use ? make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3])
                                           : make_float4(0.f, 0.f, 0.f, 0.f);
                    const uint32_t off = (uint32_t)(((split * kGvRows + r) * gpc + gi / S) * 16);
                    st_dsmem4(dsmem_map(rb + off, (uint32_t)(gi % S)), val);
                }
            }
        }
        __syncwarp();
        cluster_arrive();   // every push has landed once all have arrived
        cluster_wait();
        if (epi_warp && nok && !*(volatile int *)&s_abort) {
            // sum of group lg's S partials, in split order
            auto gsum = [&](int lg, float (&t)[4]) {
                t[0] = t[1] = t[2] = t[3] = 0.f;
                for (int sp = 0; sp < S; ++sp) {
                    const float4 p = recv[(sp * kGvRows + r) * gpc + lg];
                    t[0] += p.x;
                    t[1] += p.y;
                    t[2] += p.z;
                    t[3] += p.w;
                }
            };
#pragma unroll
            for (int lg = 0; lg < kGvResGroups; ++lg) {   // residuals loaded ahead
                const int gi = lg * S + split;
                if (lg < gpc && gi < groups) {
                    float t[4];
                    gsum(lg, t);
                    for (int j = 0; j < 4; ++j) t[j] *= scale;
                    gv_apply<EPI, 4>(a, gi * 4, mmax, n, t, bias, s_slot, nullptr,
                                     kRes ? res + 4 * lg : nullptr);
                }
            }
            for (int lg = kGvResGroups; lg < gpc; ++lg) {
                const int gi = lg * S + split;
                if (gi >= groups) break;
                float t[4];
                gsum(lg, t);
                for (int j = 0; j < 4; ++j) t[j] *= scale;
                gv_apply<EPI, 4>(a, gi * 4, mmax, n, t, bias, s_slot, nullptr);
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

int gemv_tc_box_rows_w() { return kGvRows; }

// K splits of a launch: the fewest that give at least 1.5 CTAs per SM, while
// all CTAs still fit at once (two per SM) and every split streams >= 4
// k-blocks.  Measured per matrix on GB300 (7b1 shapes, 1-32 tokens, launches
// back to back): QKV (96 row tiles) is fastest split 3 ways, the MLP up
// (128 tiles) 2 ways, the 4096-row dense and down (32 tiles) 8 ways; unsplit,
// those leave 24-120 SMs idle (QKV 23 vs 21 us, down 75 vs 28 us).
int gemv_tc_splits(int N, int K, int M, int epi, int num_sms, int int8) {
    const int nt = gemv_tc_nt(M);
    if (epi == EPI_ARGMAX || nt == 0 || nt == 256 || num_sms < 1) return 1;
    const int tiles = (N + kGvRows - 1) / kGvRows;
    const int kb = int8 ? 128 : kGvBK;   // k per stage
    const int nkb = (K + kb - 1) / kb;
    // >= 1.5 CTAs per SM; >= 1.25 for QKV, so that more SMs keep a slot for the
    // attention kernel, which starts early beside it.  Measured on GB300 (7b1,
    // 30 layers, decode step at 32 / 8 sequences): QKV in 2 splits 3.282 / 2.853 ms
    // vs 3 splits 3.298 / 2.877 (4: 3.405 / 2.967); dense in 4 / 6 / 8 splits
    // 3.336 / 3.322 / 3.298 at 32; down in 4 / 8 / 12 3.449 / 3.298 / 3.426; up
    // in 1 / 2 / 3 3.348 / 3.298 / 3.464.
    const int num = epi == EPI_QKV ? 5 : 3, den = epi == EPI_QKV ? 4 : 2;
    int s = 1;
    while (s < kGvMaxSplits && den * tiles * s < num * num_sms) ++s;
    while (s > 1 && (tiles * s > 2 * num_sms || nkb / s < kGvMinKbPerSplit)) --s;
    return s;
}

template <int EPI, int NT, bool W8>
static cudaError_t gv_configure() {
    using C = GvCfg<NT, W8>;
    cudaError_t e = cudaFuncSetAttribute(gemv_tc_kernel<EPI, NT, W8>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::Smem);
    if (e == cudaSuccess && EPI != EPI_ARGMAX && C::CanSplit)
        e = cudaFuncSetAttribute(gemv_tc_kernel<EPI, NT, W8>,
                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return e;
}

template <int EPI, int NT, bool W8>
static cudaError_t gv_launch_t(const void *mw, const void *mx, const GemvTcArgs &g, cudaStream_t s) {
    using C = GvCfg<NT, W8>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = gv_configure<EPI, NT, W8>();
        if (e != cudaSuccess) return e;
        configured = true;
    }
    if (g.splits > 1 && (!C::CanSplit || EPI == EPI_ARGMAX)) return cudaErrorInvalidValue;
    const CUtensorMap &tw = *reinterpret_cast<const CUtensorMap *>(mw);
    const CUtensorMap &tx = *reinterpret_cast<const CUtensorMap *>(mx);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((g.a.N + kGvRows - 1) / kGvRows), (unsigned)g.splits);
    cfg.blockDim = dim3(kGvThreads);
    cfg.dynamicSmemBytes = C::Smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = g_pdl ? 1 : 0;
    int na = 1;
    if (g.splits > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = 1;
        attr[1].val.clusterDim.y = (unsigned)g.splits;
        attr[1].val.clusterDim.z = 1;
        na = 2;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, gemv_tc_kernel<EPI, NT, W8>, tw, tx, g);
}

template <int EPI>
static cudaError_t gv_launch_epi(const void *mw, const void *mx, const GemvTcArgs &g, int nt,
                                 cudaStream_t s) {
    if constexpr (EPI != EPI_ARGMAX) {
        if (g.a.int8) {
            switch (nt) {   // int8 weights: up to 128 token columns (TMEM A buffers + accumulator)
                case 16: return gv_launch_t<EPI, 16, true>(mw, mx, g, s);
                case 32: return gv_launch_t<EPI, 32, true>(mw, mx, g, s);
                case 64: return gv_launch_t<EPI, 64, true>(mw, mx, g, s);
                case 128: return gv_launch_t<EPI, 128, true>(mw, mx, g, s);
                default: return cudaErrorInvalidValue;
            }
        }
    }
    switch (nt) {
        case 16: return gv_launch_t<EPI, 16, false>(mw, mx, g, s);
        case 32: return gv_launch_t<EPI, 32, false>(mw, mx, g, s);
        case 64: return gv_launch_t<EPI, 64, false>(mw, mx, g, s);
        case 128: return gv_launch_t<EPI, 128, false>(mw, mx, g, s);
        case 256: return gv_launch_t<EPI, 256, false>(mw, mx, g, s);
        default: return cudaErrorInvalidValue;
    }
}

template <int EPI>
static cudaError_t gv_prepare_epi() {
    cudaError_t e;
    if ((e = gv_configure<EPI, 16, false>())) return e;
    if ((e = gv_configure<EPI, 32, false>())) return e;
    if ((e = gv_configure<EPI, 64, false>())) return e;
    if ((e = gv_configure<EPI, 128, false>())) return e;
    if ((e = gv_configure<EPI, 256, false>())) return e;
    if constexpr (EPI != EPI_ARGMAX) {   // the LM head is always bf16
        if ((e = gv_configure<EPI, 16, true>())) return e;
        if ((e = gv_configure<EPI, 32, true>())) return e;
        if ((e = gv_configure<EPI, 64, true>())) return e;
        if ((e = gv_configure<EPI, 128, true>())) return e;
    }
    return cudaSuccess;
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
    if (a.T != 0 || gemv_tc_nt(a.M) != nt || a.M > kMaxBatch) return cudaErrorInvalidValue;
    if (a.int8 ? (a.K % 16 || !a.scale || nt > kGvInt8MaxNt || a.epi == EPI_ARGMAX) : a.K % 8)
        return cudaErrorInvalidValue;
    if (g.splits < 1 || g.splits > kGvMaxSplits || (g.splits > 1 && a.epi == EPI_ARGMAX))
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
