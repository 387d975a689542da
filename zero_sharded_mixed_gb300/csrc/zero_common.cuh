// Shared device helpers and host-side argument checks for the sm_103a kernels.
#pragma once

#include <cuda_runtime.h>
#include <cstdint>

#include "zero_gb300.h"

namespace zgb {

#ifndef ZGB_THREADS
#define ZGB_THREADS 256
#endif
constexpr int kThreads = ZGB_THREADS;   // threads per CTA for every streaming kernel

// ----------------------------------------------------------------- device

// bf16 -> fp32 is exact: the bf16 bits are the upper half of the fp32 bits.
__device__ __forceinline__ float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }
__device__ __forceinline__ float bf16_one(uint16_t x) { return __uint_as_float(((uint32_t)x) << 16); }

// Two fp32 -> packed bf16x2, round to nearest even (hardware cvt.rn);
// `lo` lands in bits 0..15 (the lower address), `hi` in bits 16..31.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ uint16_t to_bf16(float x) {
    return (uint16_t)(pack_bf16x2(x, 0.0f) & 0xffffu);
}

// 128-bit loads and stores of the streams.  Every byte of these kernels is
// touched once per launch, so nothing is worth keeping in L1; the cache
// policy is a compile-time choice (measured): ZGB_LD_HINT 1 = ld.global.cs
// (evict-first), 0 = plain ld.global, 2 = ld.global.nc (read-only path);
// ZGB_ST_HINT 1 = st.global.cs (evict-first), 0 = plain st.global.
#ifndef ZGB_LD_HINT
#define ZGB_LD_HINT 1
#endif
#ifndef ZGB_ST_HINT
#define ZGB_ST_HINT 1
#endif
__device__ __forceinline__ uint4 ld_stream_u4(const void* p) {
#if ZGB_LD_HINT == 1
    return __ldcs(reinterpret_cast<const uint4*>(p));
#elif ZGB_LD_HINT == 2
    return __ldg(reinterpret_cast<const uint4*>(p));
#else
    return *reinterpret_cast<const uint4*>(p);
#endif
}
__device__ __forceinline__ float4 ld_stream_f4(const void* p) {
#if ZGB_LD_HINT == 1
    return __ldcs(reinterpret_cast<const float4*>(p));
#elif ZGB_LD_HINT == 2
    return __ldg(reinterpret_cast<const float4*>(p));
#else
    return *reinterpret_cast<const float4*>(p);
#endif
}
__device__ __forceinline__ uint2 ld_stream_u2(const void* p) {
#if ZGB_LD_HINT == 1
    return __ldcs(reinterpret_cast<const uint2*>(p));
#elif ZGB_LD_HINT == 2
    return __ldg(reinterpret_cast<const uint2*>(p));
#else
    return *reinterpret_cast<const uint2*>(p);
#endif
}
__device__ __forceinline__ void st_stream_u4(void* p, uint4 v) {
#if ZGB_ST_HINT == 1
    __stcs(reinterpret_cast<uint4*>(p), v);
#else
    *reinterpret_cast<uint4*>(p) = v;
#endif
}
__device__ __forceinline__ void st_stream_f4(void* p, float4 v) {
#if ZGB_ST_HINT == 1
    __stcs(reinterpret_cast<float4*>(p), v);
#else
    *reinterpret_cast<float4*>(p) = v;
#endif
}

// ----------------------------------------------------------------- host

// 0 if p is device (or managed) memory of the current device, else ZERO_EINVAL.
int check_device_ptr(const void* p);
// Also 0 for pinned host memory that the device addresses at the same pointer
// (read by the kernels over the host link).
int check_source_ptr(const void* p);
// Whether a caller's layout has the shape zero_layout gives: n_dp >= 1,
// shard >= 0 and padded_n = shard * n_dp, with the product at most
// INT64_MAX / 8 (zero_layout's own limit, which keeps every byte offset in
// range) and computed only once it cannot overflow.
inline bool layout_shape_ok(const zero_layout_t* L) {
    constexpr int64_t kMaxElems = INT64_MAX / 8;
    return L->n_dp >= 1 && L->shard >= 0 && L->shard <= kMaxElems / L->n_dp &&
           L->padded_n == L->shard * (int64_t)L->n_dp;
}
// ZERO_EALIGN unless p is a multiple of `bytes`.
inline int check_aligned(const void* p, int bytes) {
    return (reinterpret_cast<uintptr_t>(p) % (uintptr_t)bytes) ? ZERO_EALIGN : ZERO_OK;
}
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
// SM count of the current device (cached per device).
int sm_count();
// CTAs of `threads` each that fit on one SM for `kernel` with `smem` bytes of
// dynamic shared memory on the current device; cached, safe from any thread.
int ctas_per_sm(const void* kernel, int threads, size_t smem);
// ZERO_ECUDA if the last launch on this thread failed (remembered for
// zero_last_cuda_error).
int launch_status();
void note_cuda_error(cudaError_t e);
const char* last_cuda_error_name();
// Grid for a grid-stride loop over `work` items with `per_cta` items per CTA
// pass, capped at `cap` CTAs (callers pass the CTAs resident at once times a
// measured number of waves).
inline unsigned grid_for(int64_t work, int64_t per_cta, int64_t cap) {
    int64_t g = (work + per_cta - 1) / per_cta;
    if (g > cap) g = cap;
    if (g < 1) g = 1;
    return (unsigned)g;
}

}  // namespace zgb
