// LM head + argmax without any allocation: the kernel's scratch lives in a
// fixed device array of this library instead of memory obtained per call.
//
// Some callers cannot allocate device memory on the call path: cudaMalloc and
// cudaFree may synchronise the device and can fail under memory pressure, a
// process may have handed all GPU memory to another framework's caching
// allocator, and latency-critical serving loops often forbid any allocation
// between requests.  bloom_op_lmhead_argmax allocates its small scratch per
// call; this variant takes no memory from the caller or the allocator at all.
#include <mutex>

#include "../../include/bloom.h"
#include "kernels.h"

using namespace bloom;

namespace {

constexpr int kNoAllocMaxRows = kMaxBatch;   // largest M the fixed scratch serves
constexpr size_t kTicketBytes = 256;         // completion ticket, padded to 256 bytes
constexpr size_t kScratchBytes = kTicketBytes + (size_t)kNoAllocMaxRows * 8;

// [0, 256): int ticket; [256, ...): unsigned long long best[kNoAllocMaxRows].
// Every GPU that loads the library holds this array until the process exits.
static __device__ __align__(256) unsigned char g_head_scratch[kScratchBytes];

std::mutex g_mu;
void *g_addr[256];   // device address of g_head_scratch, per device ordinal

// Host code may not use g_head_scratch's name as a device address (it names a
// host-side stand-in); ask the runtime once per device, with that device current.
cudaError_t scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 256) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_head_scratch);
        if (e != cudaSuccess) return e;
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" bloom_status bloom_op_lmhead_argmax_noalloc(const void *x, const void *emb, int32_t M,
                                                       int32_t V, int32_t K, int32_t *out_tokens,
                                                       float *out_logits, void *stream) {
    if (!x || !emb || !out_tokens) {
        bloom_set_error("bloom_op_lmhead_argmax_noalloc: null argument");
        return BLOOM_E_INVALID;
    }
    if (M < 1 || M > kNoAllocMaxRows) {
        bloom_set_error("bloom_op_lmhead_argmax_noalloc: M=%d rows, the fixed scratch holds 1..%d",
                        M, kNoAllocMaxRows);
        return BLOOM_E_CAPACITY;
    }
    if (V < 1 || K < 8 || K % 8) {
        bloom_set_error("bloom_op_lmhead_argmax_noalloc: V=%d K=%d (V >= 1, K >= 8, K %% 8 == 0)",
                        V, K);
        return BLOOM_E_UNSUPPORTED;
    }
    if (((uintptr_t)x & 15u) || ((uintptr_t)emb & 15u)) {
        bloom_set_error("bloom_op_lmhead_argmax_noalloc: x and emb must be 16-byte aligned");
        return BLOOM_E_INVALID;
    }
    void *scratch = nullptr;
    cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess) {
        bloom_set_error("bloom_op_lmhead_argmax_noalloc: cudaGetSymbolAddress: %s",
                        cudaGetErrorString(e));
        return BLOOM_E_CUDA;
    }
    cudaStream_t s = (cudaStream_t)stream;
    // the array keeps whatever the last call left: clear the rows this call uses
    e = cudaMemsetAsync(scratch, 0, kTicketBytes + (size_t)M * 8, s);
    if (e == cudaSuccess) {
        g_pdl = true;
        LinearArgs a;
        a.w = emb;
        a.x = (const uint16_t *)x;
        a.M = M;
        a.N = V;
        a.K = K;
        a.epi = EPI_ARGMAX;
        a.logits = out_logits;
        a.ticket = (int *)scratch;
        a.best = (unsigned long long *)((char *)scratch + kTicketBytes);
        a.out_tokens = out_tokens;
        e = launch_linear(a, bloom_device_sms(), s);
    }
    if (e != cudaSuccess) {
        bloom_set_error("bloom_op_lmhead_argmax_noalloc: %s", cudaGetErrorString(e));
        return BLOOM_E_CUDA;
    }
    return BLOOM_OK;
}
