// The 8-bit block format's arithmetic on bf16 bit patterns, shared by the
// quantizer (zero_quant.cu) and the update kernels that quantize their own
// output (zero_rs_adamw.cu).  Format ("ZeRO Optimizer, in depth", "Offload and
// ZeRO++"; reading stated in zero_gb300.h): per block, scale = max|w| / 127,
// inv = 127 / max|w| (both one IEEE division), code = round-half-even(w * inv),
// a zero block has scale 0 and codes 0.
#pragma once

#include "zero_common.cuh"

namespace zgb {

// The int8 code of x * inv (|x * inv| <= 127.00002): add 1.5 * 2^23 in fp32,
// which rounds to the nearest integer with ties to even; the low byte of the
// sum's bits holds the code in two's complement.
__device__ __forceinline__ uint32_t code_bits(float x, float inv) {
    return __float_as_uint(__fadd_rn(__fmul_rn(x, inv), 12582912.0f));
}

// Eight codes from eight bf16 weights (one 16-byte vector) packed into 8 bytes.
__device__ __forceinline__ uint2 quant8(const uint4 raw, float inv) {
    const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
    uint32_t c[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        c[2 * k] = code_bits(bf16_lo(w4[k]), inv);
        c[2 * k + 1] = code_bits(bf16_hi(w4[k]), inv);
    }
    const uint32_t lo = __byte_perm(__byte_perm(c[0], c[1], 0x0040), __byte_perm(c[2], c[3], 0x0040), 0x5410);
    const uint32_t hi = __byte_perm(__byte_perm(c[4], c[5], 0x0040), __byte_perm(c[6], c[7], 0x0040), 0x5410);
    return make_uint2(lo, hi);
}

// max over the 8 bf16 of a vector of |w|, as a pair of 16-bit lanes
__device__ __forceinline__ uint32_t absmax8_bits(const uint4 raw, uint32_t m) {
    m = __vmaxu2(m, raw.x & 0x7fff7fffu);
    m = __vmaxu2(m, raw.y & 0x7fff7fffu);
    m = __vmaxu2(m, raw.z & 0x7fff7fffu);
    return __vmaxu2(m, raw.w & 0x7fff7fffu);
}

// The block maximum of |w| from a warp whose 32 lanes each hold 8 of the
// block's 256 bf16 weights (the bits of m from absmax8_bits): one redux.sync.
// For finite values |w| orders as (bits & 0x7fff) does.
__device__ __forceinline__ float warp_block_absmax(uint32_t m) {
    m = __reduce_max_sync(0xffffffffu, (m & 0xffffu) > (m >> 16) ? (m & 0xffffu) : (m >> 16));
    return bf16_one((uint16_t)m);
}

}  // namespace zgb
