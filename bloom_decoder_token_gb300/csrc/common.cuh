// Device helpers shared by the kernels of the BLOOM decode engine (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace bloom {

constexpr int kWarp = 32;

// Device flag bits (bloom_check_device).
enum : int {
    kErrToken = 1,      // token id outside [0, vocab)
    kErrSlot = 2,       // cache slot outside [0, max_seq)
    kErrEmptyRow = 4,   // prompt row without a token
    kErrTimeout = 8,    // a bounded wait expired (results of that launch are invalid)
};

// ---- bf16 <-> f32 (bf16 is the upper half of a binary32) ----
__device__ __forceinline__ float bf_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }
__device__ __forceinline__ float bf2f(uint16_t v) { return __uint_as_float((uint32_t)v << 16); }

// Round to nearest even; NaN stays NaN.
__device__ __forceinline__ uint16_t f2bf(float f) {
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40u);
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}
__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
    return (uint32_t)f2bf(lo) | ((uint32_t)f2bf(hi) << 16);
}

// 8 bf16 in a uint4 -> 8 floats
__device__ __forceinline__ void unpack8(const uint4 &v, float *f) {
    f[0] = bf_lo(v.x); f[1] = bf_hi(v.x);
    f[2] = bf_lo(v.y); f[3] = bf_hi(v.y);
    f[4] = bf_lo(v.z); f[5] = bf_hi(v.z);
    f[6] = bf_lo(v.w); f[7] = bf_hi(v.w);
}

// ---- loads ----
// Weight stream: read once per step, so keep it out of L1.
__device__ __forceinline__ uint4 ld_stream(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}
// Activations: small, re-read by every warp of the SM; cache in L1.
__device__ __forceinline__ uint4 ld_act(const void *p) {
    return __ldg(reinterpret_cast<const uint4 *>(p));
}

// ---- asynchronous global -> shared copies (one 16-byte piece per call) ----
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

// ---- reductions ----
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Sum over a block of NW warps; every thread gets the result.  `red` holds
// NW floats of shared memory; the call contains two barriers.
template <int NW>
__device__ __forceinline__ float block_sum(float v, float *red) {
    v = warp_sum(v);
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    __syncthreads();
    if (lane == 0) red[w] = v;
    __syncthreads();
    float t = 0.f;
#pragma unroll
    for (int i = 0; i < NW; ++i) t += red[i];
    return t;
}

// Programmatic dependent launch: wait until the preceding kernel's results are
// visible / let the next kernel in the stream start launching.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;"); }

// tanh-form GeLU with the BLOOM constants; tanhf from the CUDA math library.
__device__ __forceinline__ float gelu_tanh(float x) {
    return x * 0.5f * (1.0f + tanhf(0.79788456f * x * (1.0f + 0.044715f * x * x)));
}

// Total order on float bits: larger float -> larger key (NaN above +inf).
__device__ __forceinline__ uint32_t ordered_key(float f) {
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
// (value, index) packed so that a 64-bit max picks the larger value and, on
// ties, the lower index.
__device__ __forceinline__ unsigned long long pack_argmax(float v, uint32_t idx) {
    return ((unsigned long long)ordered_key(v) << 32) | (unsigned long long)(0xffffffffu - idx);
}
__device__ __forceinline__ uint32_t unpack_index(unsigned long long p) {
    return 0xffffffffu - (uint32_t)(p & 0xffffffffull);
}

}  // namespace bloom
