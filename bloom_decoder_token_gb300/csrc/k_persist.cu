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
//  * a linear phase is a sequence of (row group of 8 rows, batch of 4 chunks
//    along K) cut into one contiguous piece per warp of the grid, equal to
//    within one batch (the stream-K split): no warp waits for another inside a
//    phase.  A warp accumulates each row group it covers and runs its fused
//    epilogue itself (Q/K/V scatter into the cache, GeLU, float32 residual
//    add, LM-head argmax -- the fusions of "DeepSpeed Inference", III.D); a row
//    group cut between consecutive warps is summed, in warp order, by the last
//    of them to finish (a ticket, no waiting), so results do not depend on
//    timing;
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
constexpr int kPXsBytes = 66 * 1024;          // staged activations of a linear phase
constexpr long long kPWaitCycles = 4000000000ll;

static_assert(kLnThreads == kPThreads, "LayerNorm rows are normalised by one whole block");

// Activations written by other blocks of this launch: coherent (L1-cached,
// invalidated by the barrier's acquire fence), never ld.global.nc.
__device__ __forceinline__ uint4 ld_coherent(const void *p) {
    return *reinterpret_cast<const uint4 *>(p);
}

// A warp's position in its weight stream: phase p, batch i of the phase (row
// group rg, batch b of the row = chunks 4b .. 4b + 3), end of its piece, and
// the lane's source address of batch i, all advanced incrementally (no
// division or 64-bit multiply per batch).  A chunk of row r is the 64 bytes at
// byte offset 64 * ch of the row (32 bf16 or 64 int8 weights); lane (g, q)
// copies bytes [16q, 16q + 16) of it for row 8 * rg + g.  Batches b < nbt_full
// lie wholly inside the row.
struct Stream {
    int p;
    long long i, end;
    int rg, b, nbt, nbt_full, N;
    int row_bytes;
    const char *w;
    const char *src;   // this lane's bytes of chunk 4b of row 8 rg + g
};

// The phases' weight streams, copied into shared memory at launch so that a
// warp crossing into the next phase never waits on global memory.
struct StreamTab {
    const PersistStream *t;
    int n;
};

// Piece of a phase of `tb` batches owned by warp `gw` of `gws`.
__device__ __forceinline__ long long piece_lo(long long tb, int gw, int gws) {
    return tb * gw / gws;
}
// The warp whose piece holds batch i.
__device__ __forceinline__ int piece_owner(long long tb, long long i, int gws) {
    return (int)(((i + 1) * gws - 1) / tb);
}

__device__ __forceinline__ void stream_row(Stream &s, int lane) {
    s.src = s.w + (size_t)(s.rg * 8 + (lane >> 2)) * s.row_bytes + (size_t)s.b * 256 + (lane & 3) * 16;
}

__device__ __forceinline__ void stream_load(const StreamTab &tab, Stream &s, int gw, int gws,
                                            int lane) {
    s.i = s.end = 0;
    if (s.p >= tab.n) return;
    const PersistStream &d = tab.t[s.p];
    if (d.tb == 0) return;
    s.i = piece_lo(d.tb, gw, gws);
    s.end = piece_lo(d.tb, gw + 1, gws);
    s.nbt = d.nbt;
    s.rg = (int)(s.i / d.nbt);
    s.b = (int)(s.i - (long long)s.rg * d.nbt);
    s.N = d.N;
    s.row_bytes = d.row_bytes;
    s.nbt_full = s.row_bytes / 256;
    s.w = d.w;
    stream_row(s, lane);
}

// Moves s to the next batch this warp streams (s itself if it is one).
__device__ __forceinline__ void stream_settle(const StreamTab &tab, Stream &s, int gw, int gws,
                                              int lane) {
    while (s.p < tab.n && s.i >= s.end) {
        ++s.p;
        stream_load(tab, s, gw, gws, lane);
    }
}

// Issue the cp.async copies of the batch at s into this lane's ring slot
// (one group, possibly empty), then advance s.
__device__ __forceinline__ void issue_batch(const StreamTab &tab, Stream &s, unsigned char *slot,
                                            int lane, int gw, int gws) {
    if (s.p < tab.n) {
        const int g = lane >> 2, q = lane & 3;
        unsigned char *dst = slot + lane * 16;
        if (s.rg * 8 + g < s.N) {
            if (s.b < s.nbt_full) {
#pragma unroll
                for (int u = 0; u < kPU; ++u) cp_async16(dst + u * kPChunk, s.src + u * 64);
            } else {
                const int off0 = s.b * 256 + q * 16;
#pragma unroll
                for (int u = 0; u < kPU; ++u)
                    if (off0 + u * 64 < s.row_bytes) cp_async16(dst + u * kPChunk, s.src + u * 64);
            }
        }
        ++s.i;
        s.src += 256;
        if (++s.b == s.nbt) {
            s.b = 0;
            ++s.rg;
            stream_row(s, lane);
        }
        if (s.i >= s.end) stream_settle(tab, s, gw, gws, lane);
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
        // arrive: a release add (no return value to wait for) publishes the
        // block's writes, ordered before it by the block barrier above
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(pa.bar) : "memory");
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

// One batch (kPU consecutive chunks): every load first (weight fragments from
// the ring slot, activations of tokens g and g+8 at xa / xb -- shared memory
// or global memory, 8 * XW bytes per chunk), then the mma steps.  FULL: every
// chunk lies inside the row; otherwise chunk u is used when u < nu and lane
// q's slice of it when kq + u * KC < K.
template <bool INT8, bool FULL>
__device__ __forceinline__ void mma_batch(float (&acc)[2][4], const unsigned char *slot,
                                          const uint16_t *xa_p, const uint16_t *xb_p, bool a_ok,
                                          bool b_ok, bool wok, int kq, int K) {
    constexpr int EPL = INT8 ? 16 : 8;
    constexpr int KC = 4 * EPL;
    constexpr int NS = EPL / 4;
    constexpr int XW = EPL / 2;
    uint4 wv[kPU];
    uint32_t xa[kPU][XW], xb[kPU][XW];
#pragma unroll
    for (int u = 0; u < kPU; ++u) {
        const bool kok = FULL || kq + u * KC < K;
        wv[u] = make_uint4(0u, 0u, 0u, 0u);
        if (wok && kok) wv[u] = *reinterpret_cast<const uint4 *>(slot + u * kPChunk);
#pragma unroll
        for (int hh = 0; hh < XW / 4; ++hh) {
            uint4 va = make_uint4(0u, 0u, 0u, 0u), vb = va;
            if (a_ok && kok) va = ld_coherent(xa_p + u * KC + 8 * hh);
            if (b_ok && kok) vb = ld_coherent(xb_p + u * KC + 8 * hh);
            xa[u][4 * hh + 0] = va.x; xa[u][4 * hh + 1] = va.y;
            xa[u][4 * hh + 2] = va.z; xa[u][4 * hh + 3] = va.w;
            xb[u][4 * hh + 0] = vb.x; xb[u][4 * hh + 1] = vb.y;
            xb[u][4 * hh + 2] = vb.z; xb[u][4 * hh + 3] = vb.w;
        }
    }
#pragma unroll
    for (int u = 0; u < kPU; ++u) {
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
            // two independent accumulator chains (even / odd chunks)
            mma_bf16_16816(acc[u & 1], xa[u][2 * s], xb[u][2 * s], xa[u][2 * s + 1],
                           xb[u][2 * s + 1], b0, b1);
        }
    }
}

// Operands of a row group's epilogue that live in global memory, loaded when
// the warp starts the row group so that the epilogue never waits on them:
// bias and int8 scale of rows 2q, 2q+1 and, for the float32 residual add, the
// residual of tokens g, g+8 at those rows (only this row group's epilogue
// writes them).
struct EpiPre {
    float bias[2], scale[2], res[2][2];
};

__device__ __forceinline__ void epi_prefetch(const LinearArgs &a, int epi, int row0, int lane,
                                             EpiPre &p) {
    const int g = lane >> 2, q = lane & 3;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int n = row0 + 2 * q + j;
        const bool nok = n < a.N;
        p.bias[j] = (a.bias && nok) ? bf2f(a.bias[n]) : 0.f;
        p.scale[j] = (a.int8 && nok) ? bf2f(a.scale[n]) : 1.f;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int m = g + 8 * half;
            p.res[half][j] =
                (epi == EPI_RESID32 && nok && m < a.M) ? a.out32[(size_t)m * a.N + n] : 0.f;
        }
    }
}

// Epilogue of one 16 x 8 accumulator tile (tokens g, g+8; rows row0 + 2q + j),
// the persistent counterpart of the weight-streaming kernel's epilogue: same
// results, operands from `p`, the cache slot of the step's token in `slot`.
template <bool INT8, int EPI>
__device__ __forceinline__ void epi_apply(const LinearArgs &a, const float (&d)[4], int row0,
                                          int lane, const EpiPre &p, int slot,
                                          unsigned long long *s_best) {
    const int g = lane >> 2, q = lane & 3;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const int m = g + 8 * half;
        if (m >= a.M) continue;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int row = row0 + 2 * q + j;
            if (row >= a.N) continue;
            float v = d[2 * half + j];
            if constexpr (INT8) v *= p.scale[j];
            v += p.bias[j];
            const size_t o = (size_t)m * a.N + row;
            if constexpr (EPI == EPI_STORE) {
                a.out[o] = f2bf(v);
            } else if constexpr (EPI == EPI_GELU) {
                a.out[o] = f2bf(gelu_tanh(v));
            } else if constexpr (EPI == EPI_RESID) {
                a.out[o] = f2bf(bf2f(a.out[o]) + v);
            } else if constexpr (EPI == EPI_RESID32) {
                a.out32[o] = p.res[half][j] + v;
            } else if constexpr (EPI == EPI_QKV) {
                const int dh = a.head_dim;
                const int hj = row / (3 * dh);
                const int cidx = (row / dh) % 3;
                const int e = row % dh;
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
                atomicMax(&s_best[m], pack_argmax(v, (uint32_t)row));
            }
        }
    }
}

template <bool INT8>
__device__ __forceinline__ void epi_dispatch(const LinearArgs &a, int epi, const float (&d)[4],
                                             int row0, int lane, const EpiPre &p, int slot,
                                             unsigned long long *s_best) {
    switch (epi) {
        case EPI_QKV: epi_apply<INT8, EPI_QKV>(a, d, row0, lane, p, slot, s_best); break;
        case EPI_RESID32: epi_apply<INT8, EPI_RESID32>(a, d, row0, lane, p, slot, s_best); break;
        case EPI_GELU: epi_apply<INT8, EPI_GELU>(a, d, row0, lane, p, slot, s_best); break;
        case EPI_STORE: epi_apply<INT8, EPI_STORE>(a, d, row0, lane, p, slot, s_best); break;
        case EPI_RESID: epi_apply<INT8, EPI_RESID>(a, d, row0, lane, p, slot, s_best); break;
        case EPI_ARGMAX: epi_apply<INT8, EPI_ARGMAX>(a, d, row0, lane, p, slot, s_best); break;
        default: break;
    }
}

// End of a row group in a warp's piece: the whole row group -> its epilogue;
// part of it -> the partial tile goes to this warp's scratch slot (0: the
// piece's first row group, 1: its last), and the last sharer to arrive sums
// the sharers' partials in warp order and runs the epilogue.
template <bool INT8>
__device__ __forceinline__ void finish_group(const PersistArgs &pa, const PersistPhase &ph, int rg,
                                             long long first_i, long long last_i,
                                             const float (&acc)[2][4], const EpiPre &pre, int slot,
                                             int lane, int gw, int gws, long long piece_first,
                                             unsigned long long *s_best) {
    const LinearArgs &a = ph.lin;
    const long long g0 = (long long)rg * ph.nbt, g1 = g0 + ph.nbt - 1;   // the group's batches
    float d[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) d[r] = acc[0][r] + acc[1][r];
    if (first_i == g0 && last_i == g1) {
        epi_dispatch<INT8>(a, a.epi, d, rg * 8, lane, pre, slot, s_best);
        return;
    }
    // sharers: the distinct owners of the group's batches, in order (pieces
    // can be empty when the phase has fewer batches than warps)
    int sharers = 0;
    for (long long i = g0; i <= g1; i = piece_lo(ph.tb, piece_owner(ph.tb, i, gws) + 1, gws))
        ++sharers;
    const int mine = (piece_first / ph.nbt == rg) ? 0 : 1;
    float *part = pa.part + ((size_t)gw * 2 + mine) * 128;
    *reinterpret_cast<float4 *>(part + lane * 4) = make_float4(d[0], d[1], d[2], d[3]);
    __syncwarp();
    int last = 0;
    if (lane == 0) {
        // acq_rel: publishes this warp's partial, and (for the last sharer)
        // orders the reads of the others' partials after their arrivals
        int old;
        asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;"
                     : "=r"(old)
                     : "l"(pa.rg_ticket + rg)
                     : "memory");
        last = old == sharers - 1;
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (!last) return;
    float t[4] = {0.f, 0.f, 0.f, 0.f};
    for (long long i = g0; i <= g1;) {
        const int w = piece_owner(ph.tb, i, gws);
        const long long wf = piece_lo(ph.tb, w, gws);
        i = piece_lo(ph.tb, w + 1, gws);
        const int sl = (wf / ph.nbt == rg) ? 0 : 1;
        const float4 v = __ldcg(reinterpret_cast<const float4 *>(pa.part + ((size_t)w * 2 + sl) * 128) + lane);
        t[0] += v.x;
        t[1] += v.y;
        t[2] += v.z;
        t[3] += v.w;
    }
    if (lane == 0) pa.rg_ticket[rg] = 0;
    epi_dispatch<INT8>(a, a.epi, t, rg * 8, lane, pre, slot, s_best);
}

// One linear phase: this warp's piece of the (row group, batch) sequence, every
// weight fragment taken from the lane's ring slot.
// Out of line (its own register allocation); the stream state is copied in and
// out so that the loop keeps it in registers.
template <bool INT8, bool XS>
__device__ __noinline__ void linear_phase(const PersistArgs &pa, const StreamTab &tab,
                                          const PersistPhase &ph, unsigned char *ring,
                                          unsigned char *xs, Stream &prod_io, unsigned &seq_io,
                                          float *s_sum, unsigned long long *s_best, int *s_last) {
    Stream prod = prod_io;
    unsigned seq = seq_io;
    const LinearArgs &a = ph.lin;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, q = lane & 3;
    const int gw = blockIdx.x * kPWarps + warp, gws = gridDim.x * kPWarps;
    const int M = a.M, N = a.N, K = a.K, epi = a.epi, nchunks = ph.nchunks, nbt = ph.nbt;
    const uint16_t *x = a.x;
    const int px = K * 2 + 64;   // 64 mod 128: two rows' fragments hit disjoint banks
    unsigned char *wring = ring + (size_t)warp * kPNB * kPU * kPChunk;

    if constexpr (XS) {
        if (a.ln_x) {
            // input LayerNorm of the float32 residual rows, straight into shared memory
            layernorm_rows_to_smem<8>(a, xs, px, s_sum, threadIdx.x, warp, lane);
        } else {
            // stage the M activation rows once for the whole phase
            const int rowv = K / 8, total = M * rowv;
            for (int i0 = threadIdx.x; i0 < total; i0 += 4 * kPThreads) {
                uint4 v[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int i = i0 + j * kPThreads;
                    if (i < total) v[j] = ld_coherent(x + (size_t)i * 8);
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int i = i0 + j * kPThreads;
                    if (i < total) {
                        const int m = i / rowv, c = i - m * rowv;
                        *reinterpret_cast<uint4 *>(xs + (size_t)m * px + (size_t)c * 16) = v[j];
                    }
                }
            }
        }
    }
    if (epi == EPI_ARGMAX)
        for (int i = threadIdx.x; i < M; i += blockDim.x) s_best[i] = 0ull;
    if (XS || epi == EPI_ARGMAX) __syncthreads();

    constexpr int KC = INT8 ? 64 : 32;   // k per chunk
    const int slot = (epi == EPI_QKV && a.len_ptr) ? *a.len_ptr : 0;   // fixed for the step
    const long long lo = piece_lo(ph.tb, gw, gws), hi = piece_lo(ph.tb, gw + 1, gws);
    const int nbt_full = (K * (INT8 ? 1 : 2)) / 256;
    const bool a_ok = g < M, b_ok = g + 8 < M;
    // activations of tokens g, g+8: staged rows (pitch px bytes) or global rows
    const uint16_t *xa0 = XS ? reinterpret_cast<const uint16_t *>(xs + (size_t)g * px) : x + (size_t)g * K;
    const uint16_t *xb0 = XS ? reinterpret_cast<const uint16_t *>(xs + (size_t)(g + 8) * px)
                             : x + (size_t)(g + 8) * K;
    const int kq = q * (INT8 ? 16 : 8);
    int rg = (int)(lo / nbt), b = (int)(lo - (long long)rg * nbt);
    for (long long i = lo; i < hi;) {
        // this warp's segment of row group rg: batches b .. bend - 1
        const int bend = (int)min((long long)nbt, (long long)b + (hi - i));
        const long long first_i = i;
        EpiPre pre;
        epi_prefetch(a, epi, rg * 8, lane, pre);
        const bool wok = rg * 8 + g < N;
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        const uint16_t *xa_p = xa0 + b * 4 * KC + kq, *xb_p = xb0 + b * 4 * KC + kq;
        for (; b < bend; ++b, ++i) {
            cp_async_wait<kPNB - 1>();   // this lane's batch `seq` has landed
            unsigned char *slot_w = wring + (size_t)(seq % kPNB) * kPU * kPChunk;
            if (b < nbt_full)
                mma_batch<INT8, true>(acc, slot_w + lane * 16, xa_p, xb_p, a_ok, b_ok, wok, 0, 0);
            else
                mma_batch<INT8, false>(acc, slot_w + lane * 16, xa_p, xb_p, a_ok, b_ok, wok,
                                       b * 4 * KC + kq, K);
            // the slot is consumed: refill it with the batch kPNB ahead
            issue_batch(tab, prod, slot_w, lane, gw, gws);
            ++seq;
            xa_p += 4 * KC;
            xb_p += 4 * KC;
        }
        finish_group<INT8>(pa, ph, rg, first_i, i - 1, acc, pre, slot, lane, gw, gws, lo, s_best);
        b = 0;
        ++rg;
    }
    if (epi == EPI_ARGMAX) argmax_publish(a, s_best, s_last, threadIdx.x, gridDim.x);
    prod_io = prod;
    seq_io = seq;
}

template <bool INT8>
__device__ __forceinline__ void linear_dispatch(const PersistArgs &pa, const StreamTab &tab,
                                                const PersistPhase &ph, unsigned char *ring,
                                                unsigned char *xs, Stream &prod, unsigned &seq,
                                                float *s_sum, unsigned long long *s_best,
                                                int *s_last) {
    if (ph.xs)
        linear_phase<INT8, true>(pa, tab, ph, ring, xs, prod, seq, s_sum, s_best, s_last);
    else
        linear_phase<INT8, false>(pa, tab, ph, ring, xs, prod, seq, s_sum, s_best, s_last);
}

// Block-wide copy of a phase descriptor (immutable) into shared memory.
__device__ __forceinline__ void copy_phase(PersistPhase &dst, const PersistPhase &src) {
    static_assert(sizeof(PersistPhase) % 16 == 0, "16-byte copies");
    const uint4 *s4 = reinterpret_cast<const uint4 *>(&src);
    uint4 *d4 = reinterpret_cast<uint4 *>(&dst);
    for (int i = threadIdx.x; i < (int)(sizeof(PersistPhase) / 16); i += blockDim.x) d4[i] = __ldg(s4 + i);
}

// The register-heavy block-level phases stay out of line, so that their
// register allocation does not constrain the linear phases' loop.
__device__ __noinline__ void ln_phase(const PersistPhase &ph, float *s_ln) {
    for (int r = blockIdx.x; r < ph.rows; r += gridDim.x)
        ln_row(ph.ln_src + (size_t)r * ph.h, ph.g, ph.b, ph.h, ph.eps, ph.ln_dst + (size_t)r * ph.h,
               s_ln);
}

__device__ __noinline__ void embed_phase(const PersistPhase &ph, int *err, float *s_ln) {
    for (int r = blockIdx.x; r < ph.rows; r += gridDim.x) {
        int tok = ph.tokens[r];
        if (tok < 0 || tok >= ph.vocab) {
            if (threadIdx.x == 0) atomicOr(err, kErrToken);
            tok = 0;
        }
        if (threadIdx.x == 0) {
            const int slot = *ph.len;
            if (slot >= 0 && slot < ph.max_seq)
                ph.pos[(size_t)r * ph.max_seq + slot] = ph.next_pos[r];
            else
                atomicOr(err, kErrSlot);
        }
        ln_row(ph.emb + (size_t)tok * ph.h, ph.g, ph.b, ph.h, ph.eps,
               ph.emb_dst + (size_t)r * ph.h, s_ln);
    }
}

__device__ __noinline__ void attn_phase(const PersistPhase &ph, unsigned char *s_attn) {
    const AttnDecodeArgs &at = ph.at;
    const int units = at.B * at.n * at.splits;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
        const int split = u % at.splits, j = (u / at.splits) % at.n;
        const int b = u / (at.splits * at.n);
        if (at.d == 64)
            attn_decode_block<64, kPThreads>(at, split, j, b,
                                             *reinterpret_cast<AttnSmem<64, kPThreads> *>(s_attn));
        else
            attn_decode_block<128, kPThreads>(at, split, j, b,
                                              *reinterpret_cast<AttnSmem<128, kPThreads> *>(s_attn));
    }
}

template <bool INT8>
__global__ void __launch_bounds__(kPThreads, 1) decode_persistent_kernel(const PersistArgs pa) {
    // dynamic: weight ring | staged activations | stream table
    extern __shared__ __align__(16) unsigned char ring[];
    unsigned char *xs = ring + kPRingBytes;
    PersistStream *s_tab = reinterpret_cast<PersistStream *>(xs + kPXsBytes);
    __shared__ __align__(16) PersistPhase s_ph[2];   // this phase and the next
    __shared__ float s_sum[3 * kPWarps];
    __shared__ unsigned long long s_best[kMaxBatch];
    __shared__ float s_ln[kLnWarps];
    __shared__ int s_flag, s_last;
    __shared__ __align__(16) unsigned char s_attn[sizeof(AttnSmem<128, kPThreads>)];

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gw = blockIdx.x * kPWarps + warp, gws = gridDim.x * kPWarps;
    unsigned char *wring = ring + (size_t)warp * kPNB * kPU * kPChunk;

    // fill the ring: the first kPNB batches of this warp's weight stream
    {
        const uint4 *src = reinterpret_cast<const uint4 *>(pa.streams);
        uint4 *dst = reinterpret_cast<uint4 *>(s_tab);
        const int n16 = pa.nphases * (int)(sizeof(PersistStream) / 16);
        for (int i = threadIdx.x; i < n16; i += blockDim.x) dst[i] = src[i];
        copy_phase(s_ph[0], pa.phases[0]);
    }
    __syncthreads();
    const StreamTab tab = {s_tab, pa.nphases};
    Stream prod;
    prod.p = 0;
    stream_load(tab, prod, gw, gws, lane);
    stream_settle(tab, prod, gw, gws, lane);
    for (int i = 0; i < kPNB; ++i)
        issue_batch(tab, prod, wring + (size_t)i * kPU * kPChunk, lane, gw, gws);
    unsigned seq = 0;
    unsigned nbar = 0;
    bool ok = true;


    for (int p = 0; p < pa.nphases && ok; ++p) {
        const PersistPhase &ph = s_ph[p & 1];
        if (ph.kind == PH_LINEAR) {
            if (ph.lin.int8) {
                if constexpr (INT8)
                    linear_dispatch<true>(pa, tab, ph, ring, xs, prod, seq, s_sum, s_best, &s_last);
            } else {
                linear_dispatch<false>(pa, tab, ph, ring, xs, prod, seq, s_sum, s_best, &s_last);
            }
        } else if (ph.kind == PH_LN) {
            ln_phase(ph, s_ln);
        } else if (ph.kind == PH_EMBED) {
            embed_phase(ph, pa.err, s_ln);
        } else if (ph.kind == PH_ATTN) {
            attn_phase(ph, s_attn);
        }
        if (p + 1 < pa.nphases) {
            copy_phase(s_ph[(p + 1) & 1], pa.phases[p + 1]);   // before the barrier: off the path
            ok = grid_barrier(pa, nbar++, &s_flag);
        }
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
    ph.nbt = (ph.nchunks + kPU - 1) / kPU;
    if (ph.nbt < 1) ph.nbt = 1;
    ph.tb = (long long)ph.tasks * ph.nbt;
    ph.xs = (long long)a.M * (a.K * 2 + 64) <= kPXsBytes;
}

// Largest dynamic shared memory the kernel can take (the per-block opt-in
// limit less its static shared memory); the stream table gets what the ring
// and the staged activations leave.
static int persist_dyn_max(bool int8) {
    int dev = 0, optin = 0;
    cudaFuncAttributes fa;
    if (cudaGetDevice(&dev) ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) ||
        cudaFuncGetAttributes(&fa, int8 ? decode_persistent_kernel<true> : decode_persistent_kernel<false>))
        return 0;
    return optin - (int)fa.sharedSizeBytes;
}

int persist_max_phases(int int8) {
    const int room = persist_dyn_max(int8) - kPRingBytes - kPXsBytes;
    return room > 0 ? room / (int)sizeof(PersistStream) : 0;
}

size_t persist_smem_bytes(int nphases) {
    return (size_t)kPRingBytes + kPXsBytes + (size_t)nphases * sizeof(PersistStream);
}

cudaError_t persist_prepare() {
    cudaError_t e = cudaFuncSetAttribute(decode_persistent_kernel<false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         persist_dyn_max(false));
    if (e) return e;
    return cudaFuncSetAttribute(decode_persistent_kernel<true>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, persist_dyn_max(true));
}

int persist_grid(int int8) {
    int dev = 0, sms = 0, coop = 0, per_sm = 0;
    if (cudaGetDevice(&dev) || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) ||
        cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev))
        return 0;
    if (!coop || persist_prepare()) return 0;
    const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &per_sm, int8 ? decode_persistent_kernel<true> : decode_persistent_kernel<false>,
        kPThreads, persist_dyn_max(int8));
    if (e || per_sm < 1 || persist_max_phases(int8) < 16) return 0;
    return sms;   // one block per SM
}

size_t persist_part_bytes(int grid) { return (size_t)grid * kPWarps * 2 * 128 * sizeof(float); }

cudaError_t launch_decode_persistent(const PersistArgs &pa, int int8, int grid, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kPThreads);
    cfg.dynamicSmemBytes = persist_smem_bytes(pa.nphases);
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
