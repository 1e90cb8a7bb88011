// ALiBi attention over the KV cache for one token per sequence: the split-KV
// decode kernel (the prefill attention is in k_attn_tc.cu).
//
// Score of key k for a query of head j:  s_k = (q . k_k) / sqrt(d) + slope_j * pos_k,
// where pos_k is the key's position counted from the sequence's first token;
// a masked key (pad slot, pos_k = -1) takes no part in the softmax (its
// probability is exactly 0), which is what the masked_fill + float32 softmax
// of "Hugging Face BLOOM Inference Optimization" (Custom CUDA Kernels) computes.
// Scores, maxima, sums and the output accumulators are float32; only K, V, q
// and the output are bf16.
#include <math.h>

#include "attn_ops.cuh"
#include "common.cuh"
#include "kernels.h"

namespace bloom {

constexpr int kAttnThreads = 128;

// ---------------------------------------------------------------------------
// Decode: one query per (sequence, head).  Grid (splits, n_head, B): each CTA
// takes one contiguous key range (attn_decode_block, which also waits for the
// previous kernel).
// ---------------------------------------------------------------------------
template <int D, int NT, int MINB>
__global__ void __launch_bounds__(NT, MINB) attn_decode_kernel(const AttnDecodeArgs a) {
    __shared__ AttnSmem<D, NT> sm;
    griddep_launch();
    attn_decode_block<D, NT>(a, blockIdx.x, blockIdx.y, blockIdx.z, sm);
}

// Three forms by grid size (measured on GB300, 7b1, 30 layers, whole decode step):
//  * 128-thread CTAs (~106 registers, about four an SM) where the whole grid is
//    resident at once;
//  * 64-thread CTAs beyond that: half the keys per round but all of the grid
//    resident together -- at 32 sequences (1024 CTAs) 3.260 ms vs 3.351 with
//    128-thread CTAs capped at 80 registers (six an SM) and 3.495 uncapped; a
//    64-register cap (eight 128-thread CTAs an SM) spills: 3.626 ms;
//  * beyond the 64-thread CTAs resident at once, over a cache in device memory,
//    the bulk-staged form (attn_decode_block_bulk): at 64 / 128 sequences 4.179 /
//    5.605 ms vs 4.230 / 5.686; at 32 sequences, where the grid fits, it lost
//    (3.307 vs 3.284: its 27 KB of shared memory keep its CTAs from starting
//    beside the QKV kernel).
constexpr int kAttnWideThreads = 64;

template <int D>
__global__ void __launch_bounds__(kAttnWideThreads, 1) attn_decode_bulk_kernel(const AttnDecodeArgs a) {
    __shared__ AttnSmemBulk<D> sm;
    griddep_launch();
    attn_decode_block_bulk<D>(a, blockIdx.x, blockIdx.y, blockIdx.z, sm);
}

int attn_decode_resident_ctas(int d, int num_sms, int wide) {
    int per_sm = 0;
    cudaError_t e;
    if (d == 128 && wide)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, attn_decode_kernel<128, kAttnWideThreads, 1>,
                                                          kAttnWideThreads, 0);
    else if (d == 128)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, attn_decode_kernel<128, kAttnThreads, 1>,
                                                          kAttnThreads, 0);
    else
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, attn_decode_kernel<64, kAttnThreads, 1>,
                                                          kAttnThreads, 0);
    return e == cudaSuccess ? per_sm * num_sms : 0;
}

cudaError_t launch_attn_decode(const AttnDecodeArgs &a, cudaStream_t s) {
    dim3 grid(a.splits, a.n, a.B);
    if (a.d == 64) return launch_pdl(attn_decode_kernel<64, kAttnThreads, 1>, grid, dim3(kAttnThreads), s, a);
    if (a.d == 128) {
        const long long ctas = (long long)a.splits * a.n * a.B;
        if (ctas > a.resident_wide && a.bulk)
            return launch_pdl(attn_decode_bulk_kernel<128>, grid, dim3(kAttnWideThreads), s, a);
        if (ctas > a.resident_ctas)
            return launch_pdl(attn_decode_kernel<128, kAttnWideThreads, 1>, grid, dim3(kAttnWideThreads), s, a);
        return launch_pdl(attn_decode_kernel<128, kAttnThreads, 1>, grid, dim3(kAttnThreads), s, a);
    }
    return cudaErrorInvalidValue;
}

}  // namespace bloom
