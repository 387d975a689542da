// 8-bit quantized weight gather for stage 3 (ZeRO++), sm_103a.
//
// "ZeRO Optimizer, in depth", "Offload and ZeRO++": zero_quantized_weights
// quantises the weight all-gather; "ZeRO and FSDP", "Fewer bytes on the wire":
// the weight all-gather is quantized to 8 bits.  Each owner quantizes its own
// bf16 shard in blocks of `block` consecutive elements (symmetric int8, one
// fp32 scale per block: scale = max|w| / 127; q = round-half-even(w * inv)
// with inv = 127 / max|w|, clamped to [-127, 127]; a zero block has scale 0),
// and the gather rebuilds the full bf16 unit as bf16_rne(q * scale).  A
// receiver then reads 1 byte per weight plus 4 bytes per block instead of 2.
//
// zero_quantize_int8: a group of lanes quantizes one block (8 lanes for a
//   256-element block, four blocks per warp; 16 for 512; the whole warp for
//   1024 and 2048), each lane four or eight 8-element vectors of it, loads
//   first.  The block maximum of |w| is taken on the bf16 bit patterns: for
//   finite values |w| orders as (bits & 0x7fff) does, so two elements go
//   through one SIMD max (vmax2), and the group finishes with xor-shuffles.
//   Each element is then one multiply by inv and one add of 1.5 * 2^23, which
//   rounds to the nearest integer, ties to even (the sum lies in [2^23, 2^24)
//   where fp32 spacing is 1); the low byte of the sum's bits is the int8
//   code.  |w * inv| <= 127 * (1 + 2^-23), so no clamp is needed.  About five
//   instructions per element; 2 bytes read + 1 byte written (+4 per block).
// zero_gather_layer_int8: blockIdx.y picks the shard; a grid-stride loop over
//   8-element vectors (four per thread and iteration, loads first) loads 8
//   int8 values and their block's scale, multiplies in fp32 and stores 8 bf16
//   (cvt.rn.bf16x2).  1 byte read + 2 written per element (+ the scales).
#include "zero_quant.cuh"

#ifndef ZGB_QUANT_WAVES
#define ZGB_QUANT_WAVES 512  // grid = resident CTAs x this, quantize: in effect one pass per
                             // warp (measured: 6.9 TB/s against 5.5 at x1 and 6.4 at x16)
#endif
#ifndef ZGB_DEQUANT_WAVES
#define ZGB_DEQUANT_WAVES 64 // the same for the int8 gather (measured +17 % over x1)
#endif

namespace zgb {

constexpr int kWarps = kThreads / 32;

struct QuantParams {
    const uint16_t* w;   // n_dp shards of S bf16, back to back
    int8_t* q;           // same layout
    float* scales;       // n_dp x blocks_per_shard
    int64_t shard;       // S
    int64_t blocks_per_shard;
    int64_t total_blocks;
    int32_t block;
};

__device__ __forceinline__ int8_t quant_one(float x, float amax) {
    if (amax == 0.0f) return 0;
    return (int8_t)(code_bits(x, __fdiv_rn(127.0f, amax)) & 0xffu);
}

// A group of G lanes quantizes one block of 8 * G * V elements: each lane
// holds V 8-element vectors of it (lane l of the group: vectors l, l + G, ...),
// so a warp works on 32 / G blocks at once.  The block maximum goes through
// log2(G) xor-shuffles inside the group, and the warp issues the two IEEE
// divisions (scale and inverse) once for all of its blocks.  blockIdx.y is
// the shard (no division by the shard's block count); warps take groups of
// 32 / G consecutive blocks in a grid-stride loop.
template <int G, int V>
__global__ void __launch_bounds__(kThreads) quantize_group_kernel(const __grid_constant__ QuantParams p,
                                                                  int32_t shard0) {
    constexpr int kBlocksPerWarp = 32 / G;
    const int lane = threadIdx.x & 31;
    const int gl = lane % G;                                   // lane within its group
    const int64_t o = (int64_t)shard0 + blockIdx.y;
    const uint16_t* w = p.w + o * p.shard;
    int8_t* q = p.q + o * p.shard;
    float* sc = p.scales + o * p.blocks_per_shard;
    const int64_t warp = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    const int64_t step = (int64_t)gridDim.x * kWarps * kBlocksPerWarp;
    for (int64_t b = warp * kBlocksPerWarp + lane / G; b - lane / G < p.blocks_per_shard; b += step) {
        const int64_t k0 = b * (8 * G * V);
        const int64_t len = b < p.blocks_per_shard ? min((int64_t)(8 * G * V), p.shard - k0) : 0;
        uint4 raw[V];
        uint32_t m = 0u;
#pragma unroll
        for (int j = 0; j < V; ++j) {
            const int64_t off = (int64_t)(j * G + gl) * 8;
            if (off < len) raw[j] = ld_stream_u4(w + k0 + off);
        }
#pragma unroll
        for (int j = 0; j < V; ++j)
            if ((int64_t)(j * G + gl) * 8 < len) m = absmax8_bits(raw[j], m);
        m = (m & 0xffffu) > (m >> 16) ? (m & 0xffffu) : (m >> 16);
#pragma unroll
        for (int d = G / 2; d > 0; d /= 2) {                    // every lane of the warp takes part
            const uint32_t other = __shfl_xor_sync(0xffffffffu, m, d);
            m = other > m ? other : m;
        }
        const float a = bf16_one((uint16_t)m);
        const float scale = __fdiv_rn(a, 127.0f);
        const float inv = a == 0.0f ? 0.0f : __fdiv_rn(127.0f, a);   // a zero block: codes 0
        if (len > 0 && gl == 0) sc[b] = scale;
#pragma unroll
        for (int j = 0; j < V; ++j) {
            const int64_t off = (int64_t)(j * G + gl) * 8;
            if (off < len) *reinterpret_cast<uint2*>(q + k0 + off) = quant8(raw[j], inv);
        }
    }
}

// One thread per quantization block: ragged shards and unaligned buffers.
__global__ void __launch_bounds__(kThreads) quantize_scalar_kernel(const __grid_constant__ QuantParams p) {
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    for (int64_t qb = (int64_t)blockIdx.x * kThreads + threadIdx.x; qb < p.total_blocks; qb += stride) {
        const int64_t o = qb / p.blocks_per_shard;
        const int64_t b = qb - o * p.blocks_per_shard;
        const int64_t k0 = b * p.block;
        const int64_t len = min((int64_t)p.block, p.shard - k0);
        const int64_t base = o * p.shard + k0;
        float amax = 0.0f;
        for (int64_t i = 0; i < len; ++i) amax = fmaxf(amax, fabsf(bf16_one(p.w[base + i])));
        p.scales[o * p.blocks_per_shard + b] = __fdiv_rn(amax, 127.0f);
        for (int64_t i = 0; i < len; ++i) p.q[base + i] = quant_one(bf16_one(p.w[base + i]), amax);
    }
}

struct DequantParams {
    const int8_t* q[ZERO_MAX_SRC];
    const float* scales[ZERO_MAX_SRC];
    uint16_t* out;       // the first of these shards' places in the full buffer
    int64_t shard;
    int32_t block;
    int32_t block_shift; // log2(block): the block of element k is k >> block_shift
};

__device__ __forceinline__ uint4 dequant8(const uint2 raw, const float s) {
    const uint32_t w2[2] = {raw.x, raw.y};
    uint32_t o4[4];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const float f0 = (float)(int8_t)(w2[h] & 0xffu);
        const float f1 = (float)(int8_t)((w2[h] >> 8) & 0xffu);
        const float f2 = (float)(int8_t)((w2[h] >> 16) & 0xffu);
        const float f3 = (float)(int8_t)(w2[h] >> 24);
        o4[2 * h] = pack_bf16x2(__fmul_rn(f0, s), __fmul_rn(f1, s));
        o4[2 * h + 1] = pack_bf16x2(__fmul_rn(f2, s), __fmul_rn(f3, s));
    }
    return make_uint4(o4[0], o4[1], o4[2], o4[3]);
}

// Four 8-element vectors per thread and iteration, loads first.
__global__ void __launch_bounds__(kThreads) dequant_gather_vec_kernel(const __grid_constant__ DequantParams p) {
    constexpr int U = 4;
    const int8_t* q = p.q[blockIdx.y];
    const float* sc = p.scales[blockIdx.y];
    uint16_t* dst = p.out + (int64_t)blockIdx.y * p.shard;
    const int64_t nv = p.shard >> 3;
    const int64_t chunk = (int64_t)U * kThreads;          // consecutive vectors per CTA and pass
    for (int64_t vi = (int64_t)blockIdx.x * chunk + threadIdx.x; vi < nv; vi += (int64_t)gridDim.x * chunk) {
        uint2 raw[U];
        float s[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t k = (vi + u * kThreads) * 8;
            if (vi + u * kThreads < nv) {
                raw[u] = __ldcs(reinterpret_cast<const uint2*>(q + k));
                s[u] = __ldg(sc + (k >> p.block_shift));             // one block: block % 8 == 0
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (vi + u * kThreads < nv) st_stream_u4(dst + (vi + u * kThreads) * 8, dequant8(raw[u], s[u]));
    }
}

__global__ void __launch_bounds__(kThreads) dequant_gather_scalar_kernel(const __grid_constant__ DequantParams p) {
    const int8_t* q = p.q[blockIdx.y];
    const float* sc = p.scales[blockIdx.y];
    uint16_t* dst = p.out + (int64_t)blockIdx.y * p.shard;
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    for (int64_t k = (int64_t)blockIdx.x * kThreads + threadIdx.x; k < p.shard; k += stride)
        dst[k] = to_bf16(__fmul_rn((float)q[k], sc[k >> p.block_shift]));
}

bool valid_block(int32_t block) {
    return block >= 256 && block <= 2048 && block % 256 == 0 && (block & (block - 1)) == 0;
}

}  // namespace zgb

extern "C" int zero_quantize_int8(const zero_layout_t* unit, const uint16_t* shards_bf16, int8_t* q,
                                  float* scales, int32_t block, void* stream) {
    using namespace zgb;
    if (!unit || !shards_bf16 || !q || !scales) return ZERO_EINVAL;
    if (!valid_block(block)) return ZERO_EINVAL;
    if (!layout_shape_ok(unit))
        return ZERO_EINVAL;
    if (check_aligned(shards_bf16, 2) || check_aligned(scales, 4)) return ZERO_EALIGN;
    if (unit->shard == 0) return ZERO_OK;
    if (check_device_ptr(shards_bf16) || check_device_ptr(q) || check_device_ptr(scales))
        return ZERO_EINVAL;
    QuantParams p;
    p.w = shards_bf16;
    p.q = q;
    p.scales = scales;
    p.shard = unit->shard;
    p.block = block;
    p.blocks_per_shard = (unit->shard + block - 1) / block;
    p.total_blocks = p.blocks_per_shard * unit->n_dp;
    const bool vec = unit->shard % 8 == 0 && aligned16(shards_bf16) &&
                     (reinterpret_cast<uintptr_t>(q) & 7u) == 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (!vec) {
        const int occ = ctas_per_sm((const void*)quantize_scalar_kernel, kThreads, 0);
        quantize_scalar_kernel<<<grid_for(p.total_blocks, kThreads, (int64_t)sm_count() * occ), kThreads, 0, s>>>(p);
        return launch_status();
    }
    // 8 lanes per 256-element block (four blocks per warp), 16 per 512, 32 per
    // 1024 and 2048; four (2048: eight) vectors per lane
    const void* fns[4] = {(const void*)quantize_group_kernel<8, 4>, (const void*)quantize_group_kernel<16, 4>,
                          (const void*)quantize_group_kernel<32, 4>, (const void*)quantize_group_kernel<32, 8>};
    const int which = block == 256 ? 0 : block == 512 ? 1 : block == 1024 ? 2 : 3;
    const int occ = ctas_per_sm(fns[which], kThreads, 0);
    const int64_t per_cta = (int64_t)kWarps * (which == 0 ? 4 : which == 1 ? 2 : 1);
    const int64_t resident = (int64_t)sm_count() * occ * ZGB_QUANT_WAVES;
    for (int64_t o0 = 0; o0 < unit->n_dp; o0 += 65535) {
        const int cnt = (int)(unit->n_dp - o0 < 65535 ? unit->n_dp - o0 : 65535);
        const int64_t per_shard = resident / cnt > 0 ? resident / cnt : 1;
        const dim3 grid(grid_for(p.blocks_per_shard, per_cta, per_shard), cnt);
        switch (which) {
            case 0: quantize_group_kernel<8, 4><<<grid, kThreads, 0, s>>>(p, (int32_t)o0); break;
            case 1: quantize_group_kernel<16, 4><<<grid, kThreads, 0, s>>>(p, (int32_t)o0); break;
            case 2: quantize_group_kernel<32, 4><<<grid, kThreads, 0, s>>>(p, (int32_t)o0); break;
            default: quantize_group_kernel<32, 8><<<grid, kThreads, 0, s>>>(p, (int32_t)o0); break;
        }
        const int rc = launch_status();
        if (rc) return rc;
    }
    return ZERO_OK;
}

extern "C" int zero_gather_layer_int8(const zero_layout_t* unit, const int8_t* const* q_shards,
                                      const float* const* scale_shards, int32_t block,
                                      uint16_t* full_out, void* stream) {
    using namespace zgb;
    if (!unit || !q_shards || !scale_shards || !full_out) return ZERO_EINVAL;
    if (!valid_block(block)) return ZERO_EINVAL;
    if (!layout_shape_ok(unit))
        return ZERO_EINVAL;
    const int n_dp = unit->n_dp;
    for (int o = 0; o < n_dp; ++o)
        if (!q_shards[o] || !scale_shards[o]) return ZERO_EINVAL;
    for (int o = 0; o < n_dp; ++o)
        if (check_aligned(scale_shards[o], 4)) return ZERO_EALIGN;
    if (check_aligned(full_out, 2)) return ZERO_EALIGN;
    if (unit->shard == 0) return ZERO_OK;
    for (int o = 0; o < n_dp; ++o)
        if (check_device_ptr(q_shards[o]) || check_device_ptr(scale_shards[o])) return ZERO_EINVAL;
    if (check_device_ptr(full_out)) return ZERO_EINVAL;
    const int occ_vec = ctas_per_sm((const void*)dequant_gather_vec_kernel, kThreads, 0);
    const int occ_scalar = ctas_per_sm((const void*)dequant_gather_scalar_kernel, kThreads, 0);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    for (int o0 = 0; o0 < n_dp; o0 += ZERO_MAX_SRC) {
        const int cnt = n_dp - o0 < ZERO_MAX_SRC ? n_dp - o0 : ZERO_MAX_SRC;
        DequantParams p;
        bool vec = unit->shard % 8 == 0;
        for (int k = 0; k < ZERO_MAX_SRC; ++k) {
            p.q[k] = nullptr;
            p.scales[k] = nullptr;
        }
        for (int k = 0; k < cnt; ++k) {
            p.q[k] = q_shards[o0 + k];
            p.scales[k] = scale_shards[o0 + k];
            vec = vec && (reinterpret_cast<uintptr_t>(p.q[k]) & 7u) == 0;
        }
        p.out = full_out + (int64_t)o0 * unit->shard;
        p.shard = unit->shard;
        p.block = block;
        p.block_shift = 0;
        while ((1 << p.block_shift) < block) ++p.block_shift;   // block is a power of two
        vec = vec && aligned16(p.out);
        const int64_t resident = (int64_t)sm_count() * (vec ? occ_vec * ZGB_DEQUANT_WAVES : occ_scalar);
        const int64_t per_shard = resident / cnt > 0 ? resident / cnt : 1;
        dim3 grid(grid_for(vec ? unit->shard >> 3 : unit->shard, vec ? 4 * kThreads : kThreads, per_shard), cnt);
        if (vec)
            dequant_gather_vec_kernel<<<grid, kThreads, 0, s>>>(p);
        else
            dequant_gather_scalar_kernel<<<grid, kThreads, 0, s>>>(p);
        const int rc = launch_status();
        if (rc) return rc;
    }
    return ZERO_OK;
}
