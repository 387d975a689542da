// Stage-3 per-unit all-gather of bf16 weight shards into one full buffer, sm_103a.
//
// "DeepSpeed ZeRO", "Stage 3 step by step": before a layer runs forward (and
// again in backward) the ranks all-gather that layer's parameters, then release
// them.  "ZeRO and FSDP", "FSDP, ZeRO-3 inside PyTorch": each unit is one flat
// buffer, so gathering it is one all-gather; at most two units are resident.
//
// A pure copy: full[o*S + k] = shard_o[k].  blockIdx.y picks the shard, a
// grid-stride loop over 8-element (128-bit) vectors copies it.  2 bytes read +
// 2 bytes written per unit element.
#include "zero_common.cuh"

#ifndef ZGB_GATHER_WAVES
#define ZGB_GATHER_WAVES 16  // grid = resident CTAs x this (measured on GB300: x16 1 % over x8
                             // and x32, 3 % over x4)
#endif
#ifndef ZGB_GATHER_U
#define ZGB_GATHER_U 1       // 128-bit vectors per thread and iteration (1 measured best)
#endif

namespace zgb {

struct GatherParams {
    const uint16_t* shard[ZERO_MAX_SRC];
    uint16_t* out;      // points at the first of these shards' places in the full buffer
    int64_t shard_len;  // S
};

__global__ void __launch_bounds__(kThreads) gather_vec_kernel(const __grid_constant__ GatherParams p) {
    const uint16_t* src = p.shard[blockIdx.y];
    uint16_t* dst = p.out + (int64_t)blockIdx.y * p.shard_len;
    const int64_t nv = p.shard_len >> 3;
    const int64_t tid = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    // U vectors per thread and iteration, loads first
    constexpr int U = ZGB_GATHER_U;
    for (int64_t vi = tid; vi < nv; vi += U * stride) {
        uint4 x[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (vi + u * stride < nv) x[u] = ld_stream_u4(src + (vi + u * stride) * 8);
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (vi + u * stride < nv) st_stream_u4(dst + (vi + u * stride) * 8, x[u]);
    }
    const int64_t tail = p.shard_len - (nv << 3);
    if (tid < tail) dst[(nv << 3) + tid] = src[(nv << 3) + tid];
}

__global__ void __launch_bounds__(kThreads) gather_scalar_kernel(const __grid_constant__ GatherParams p) {
    const uint16_t* src = p.shard[blockIdx.y];
    uint16_t* dst = p.out + (int64_t)blockIdx.y * p.shard_len;
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < p.shard_len; i += stride)
        dst[i] = src[i];
}

}  // namespace zgb

extern "C" int zero_gather_layer(const zero_layout_t* unit, const uint16_t* const* shards,
                                 uint16_t* full_out, void* stream) {
    using namespace zgb;
    if (!unit || !shards || !full_out) return ZERO_EINVAL;
    if (!layout_shape_ok(unit))
        return ZERO_EINVAL;
    const int n_dp = unit->n_dp;
    for (int o = 0; o < n_dp; ++o)
        if (!shards[o]) return ZERO_EINVAL;
    for (int o = 0; o < n_dp; ++o)
        if (check_aligned(shards[o], 2)) return ZERO_EALIGN;
    if (check_aligned(full_out, 2)) return ZERO_EALIGN;
    if (unit->shard == 0) return ZERO_OK;
    for (int o = 0; o < n_dp; ++o)
        if (check_device_ptr(shards[o])) return ZERO_EINVAL;
    if (check_device_ptr(full_out)) return ZERO_EINVAL;

    const int occ_vec = ctas_per_sm((const void*)gather_vec_kernel, kThreads, 0);
    const int occ_scalar = ctas_per_sm((const void*)gather_scalar_kernel, kThreads, 0);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // shards go in groups of at most ZERO_MAX_SRC per launch (kernel parameter space)
    for (int o0 = 0; o0 < n_dp; o0 += ZERO_MAX_SRC) {
        const int cnt = n_dp - o0 < ZERO_MAX_SRC ? n_dp - o0 : ZERO_MAX_SRC;
        GatherParams p;
        bool vec = (unit->shard % 8) == 0;
        for (int k = 0; k < ZERO_MAX_SRC; ++k) p.shard[k] = nullptr;
        for (int k = 0; k < cnt; ++k) {
            p.shard[k] = shards[o0 + k];
            vec = vec && aligned16(p.shard[k]);
        }
        p.out = full_out + (int64_t)o0 * unit->shard;
        p.shard_len = unit->shard;
        vec = vec && aligned16(p.out);
        const int64_t resident = (int64_t)sm_count() * (vec ? occ_vec : occ_scalar) * ZGB_GATHER_WAVES;
        const int64_t per_shard = resident / cnt > 0 ? resident / cnt : 1;
        dim3 grid(grid_for(vec ? unit->shard >> 3 : unit->shard, kThreads, per_shard), cnt);
        if (vec)
            gather_vec_kernel<<<grid, kThreads, 0, s>>>(p);
        else
            gather_scalar_kernel<<<grid, kThreads, 0, s>>>(p);
        const int rc = launch_status();
        if (rc) return rc;
    }
    return ZERO_OK;
}
