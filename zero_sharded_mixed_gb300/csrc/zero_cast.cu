// fp32 -> bf16 cast of a weight vector, sm_103a.
//
// "ZeRO and FSDP", "The idea, one stage at a time": after the owners update
// their fp32 master shards they cast them to bf16 and all-gather the result, so
// that every rank holds the full bf16 weights.  The fused update does that cast
// for every step; this kernel does it on its own, for the first bf16 weights
// made from freshly initialised master weights and for bf16 weights rebuilt
// from restored master weights.
//
// dst[i] = RNE(src[i]) for i in [0, n): round to nearest, ties to even, by the
// hardware convert (cvt.rn.bf16x2.f32), which rounds values at or past the
// largest finite bf16 plus half an ulp to infinity and keeps subnormals.  A NaN
// keeps its sign and its top payload bits and is made quiet (the upper half of
// its bits with the quiet bit set), which fixes the result the convert leaves
// open.  A streaming pass: 4 bytes read + 2 bytes written per element, eight
// elements (two 128-bit loads, one 128-bit store) per thread and iteration.
#include "zero_common.cuh"

#ifndef ZGB_CAST_WAVES
#define ZGB_CAST_WAVES 16    // grid = resident CTAs x this, as for the gather
#endif

namespace zgb {

__device__ __forceinline__ uint32_t nan_bf16(float x) { return (__float_as_uint(x) >> 16) | 0x40u; }

// Two fp32 -> packed bf16x2 (lo in bits 0..15), NaNs fixed as above.
__device__ __forceinline__ uint32_t cast_pair(float lo, float hi) {
    uint32_t r = pack_bf16x2(lo, hi);
    if (lo != lo) r = (r & 0xffff0000u) | (nan_bf16(lo) & 0xffffu);
    if (hi != hi) r = (r & 0x0000ffffu) | (nan_bf16(hi) << 16);
    return r;
}

__device__ __forceinline__ uint16_t cast_one(float x) {
    return x != x ? (uint16_t)nan_bf16(x) : to_bf16(x);
}

__global__ void __launch_bounds__(kThreads)
cast_bf16_vec_kernel(const float* __restrict__ src, uint16_t* __restrict__ dst, int64_t n) {
    const int64_t nv = n >> 3;
    const int64_t tid = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    for (int64_t vi = tid; vi < nv; vi += stride) {
        const float4 a = ld_stream_f4(src + vi * 8);
        const float4 b = ld_stream_f4(src + vi * 8 + 4);
        uint4 o;
        o.x = cast_pair(a.x, a.y);
        o.y = cast_pair(a.z, a.w);
        o.z = cast_pair(b.x, b.y);
        o.w = cast_pair(b.z, b.w);
        st_stream_u4(dst + vi * 8, o);
    }
    const int64_t tail = n - (nv << 3);
    if (tid < tail) dst[(nv << 3) + tid] = cast_one(src[(nv << 3) + tid]);
}

__global__ void __launch_bounds__(kThreads)
cast_bf16_scalar_kernel(const float* __restrict__ src, uint16_t* __restrict__ dst, int64_t n) {
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < n; i += stride)
        dst[i] = cast_one(src[i]);
}

}  // namespace zgb

extern "C" int zero_cast_bf16(const float* src, uint16_t* dst, int64_t n, void* stream) {
    using namespace zgb;
    if (n < 0) return ZERO_EINVAL;
    if (!src || !dst) return ZERO_EINVAL;
    if (check_aligned(src, 4) || check_aligned(dst, 2)) return ZERO_EALIGN;
    if (n == 0) return ZERO_OK;
    if (check_device_ptr(src) || check_device_ptr(dst)) return ZERO_EINVAL;
    const bool vec = aligned16(src) && aligned16(dst);
    const void* kernel = vec ? (const void*)cast_bf16_vec_kernel : (const void*)cast_bf16_scalar_kernel;
    const int64_t resident = (int64_t)sm_count() * ctas_per_sm(kernel, kThreads, 0) * ZGB_CAST_WAVES;
    const unsigned grid = grid_for(vec ? n >> 3 : n, kThreads, resident);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (vec)
        cast_bf16_vec_kernel<<<grid, kThreads, 0, s>>>(src, dst, n);
    else
        cast_bf16_scalar_kernel<<<grid, kThreads, 0, s>>>(src, dst, n);
    return launch_status();
}
