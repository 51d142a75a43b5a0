// Internal helpers shared by the libpkv kernels (device primitives, status plumbing).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

// ---------------------------------------------------------------- host side
// Records a one-line reason for the status about to be returned (thread-local).
pkv_status fail(pkv_status st, const char *fmt, ...);
pkv_status ok();
// Converts the last CUDA launch error into PKV_ERR_CUDA.
pkv_status check_launch(const char *what);
// Streaming multiprocessors of the current device (cached per device).
int sm_count();

inline bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
inline bool is_pow2(int64_t x) { return x > 0 && (x & (x - 1)) == 0; }
inline int ilog2(int64_t x) {
    int s = 0;
    while ((int64_t(1) << s) < x) ++s;
    return s;
}

// ---------------------------------------------------------------- device side
__device__ __forceinline__ void raise_flag(int32_t *err, int bits) { atomicOr(err, bits); }

// 16-byte global->shared copy; src_bytes = 0 zero-fills the destination without reading.
__device__ __forceinline__ void cp_async_16(void *smem_dst, const void *gmem_src, int src_bytes) {
    const unsigned dst = static_cast<unsigned>(__cvta_generic_to_shared(smem_dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(gmem_src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// bf16 is the upper half of an fp32: widening is a shift or a mask.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ void widen8(const uint4 &r, float f[8]) {
    f[0] = bf16_lo(r.x); f[1] = bf16_hi(r.x);
    f[2] = bf16_lo(r.y); f[3] = bf16_hi(r.y);
    f[4] = bf16_lo(r.z); f[5] = bf16_hi(r.z);
    f[6] = bf16_lo(r.w); f[7] = bf16_hi(r.w);
}

// Streaming 16-byte load that does not allocate in L1.
__device__ __forceinline__ uint4 ld_stream_16(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}
__device__ __forceinline__ void st_stream_16(void *p, const uint4 &r) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};\n" ::"l"(p), "r"(r.x), "r"(r.y), "r"(r.z), "r"(r.w)
                 : "memory");
}

// Sum of v over the block (blockDim.x a multiple of 32, <= 1024); every thread gets the total.
__device__ __forceinline__ long long block_sum(long long v, long long *scratch32) {
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) scratch32[warp] = v;
    __syncthreads();
    long long t = 0;
    const int nw = blockDim.x >> 5;
    for (int i = 0; i < nw; ++i) t += scratch32[i];
    return t;
}

}  // namespace pkv
