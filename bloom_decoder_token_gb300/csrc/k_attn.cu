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
// takes one contiguous key range (attn_decode_block).
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kAttnThreads) attn_decode_kernel(const AttnDecodeArgs a) {
    __shared__ AttnSmem<D, kAttnThreads> sm;
    griddep_launch();
    griddep_wait();
    attn_decode_block<D, kAttnThreads>(a, blockIdx.x, blockIdx.y, blockIdx.z, sm);
}

cudaError_t launch_attn_decode(const AttnDecodeArgs &a, cudaStream_t s) {
    dim3 grid(a.splits, a.n, a.B);
    if (a.d == 64) return launch_pdl(attn_decode_kernel<64>, grid, dim3(kAttnThreads), s, a);
    if (a.d == 128) return launch_pdl(attn_decode_kernel<128>, grid, dim3(kAttnThreads), s, a);
    return cudaErrorInvalidValue;
}

}  // namespace bloom
