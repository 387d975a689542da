// The fused update for bf16 gradient sources with TMA staging, sm_103a: an
// opt-in alternative to the register-staged kernel (ZGB_RS_TMA=1), which it
// trails by about 5 % on GB300 (6.7 against 7.0 TB/s at GPT-2-XL sizes).
//
// Same computation as rs_adamw_vec_kernel<kPlainBf16, NDP> (zero_rs_adamw.cu):
// g = (sum over ranks of the bf16 gradients, fp32, ascending) / divisor, the
// AdamW update, the bf16 cast, the gather write -- bit-identical to it.  The
// difference is how bytes reach the SM: instead of each thread issuing its own
// 128-bit loads, one thread per CTA issues 1-D bulk copies (cp.async.bulk,
// the TMA engine's linear mode) of whole tiles -- 2 bytes per gradient element
// and 4 per state element -- into a ring of shared-memory stages, each stage
// completed by an mbarrier transaction count.  Consumers read the tile from
// shared memory, compute, and store the results straight to global memory.
// CTA b takes tiles b, b + grid, ... so the CTAs in flight work on
// neighbouring tiles.  Two designs:
//   rs_adamw_ws_kernel (default, ZGB_TMA_WS=1): warp-specialized -- a producer
//     warp and consumer warps synchronised per stage by full/empty mbarriers;
//   rs_adamw_tma_kernel (ZGB_TMA_WS=0): every thread of the CTA waits for a
//     stage, computes, and the CTA synchronises before the stage is refilled.
//
// Every wait is bounded: an mbarrier wait gives up after about one second of
// SM clock, records ZERO_ETIMEOUT in a device status word (read by
// zero_status_check), and the waiting warp or CTA stops; before the CTA ends,
// the thread that issued copies waits -- bounded again -- for those still in
// flight.  No path waits forever.
#include <cmath>

#include "zero_tma.cuh"
#include "zero_update.cuh"

#ifndef ZGB_TMA_INTERLEAVE
#define ZGB_TMA_INTERLEAVE 1   // 1: CTA b takes tiles b, b + grid, ...; 0: a contiguous run per CTA
#endif
#ifndef ZGB_TMA_STAGES
#define ZGB_TMA_STAGES 3
#endif
#ifndef ZGB_TMA_WS
#define ZGB_TMA_WS 1           // 1: the warp-specialized pipeline; 0: the CTA-synchronous ring
#endif
#ifndef ZGB_WS_STAGES
#define ZGB_WS_STAGES 2        // stages of the warp-specialized ring per CTA (measured: 2 stages at
                               // three CTAs per SM beat 3-8 stages at one or two CTAs)
#endif
#ifndef ZGB_WS_CONSUMERS
#define ZGB_WS_CONSUMERS 8     // consumer warps of the warp-specialized kernel (tile = 128 x this)
#endif
#ifndef ZGB_TMA_TIMEOUT_CYCLES
#define ZGB_TMA_TIMEOUT_CYCLES (1ll << 31)   // SM cycles before a wait gives up (~1 s)
#endif

namespace zgb {

__device__ int g_device_status;   // ZERO_OK, or ZERO_ETIMEOUT once a bounded wait gave up

constexpr int kTmaThreads = 256;
constexpr int kTile = 4 * kTmaThreads;   // elements per stage: 4 per thread
constexpr int kStages = ZGB_TMA_STAGES;
// A 4-stage ring (112 KB per CTA at 8 sources) was built once and its launch
// failed with a CUDA runtime error whose cause was not found; only the
// configurations that have run are allowed.
static_assert(kStages >= 2 && kStages <= 3, "the TMA ring runs with 2 or 3 stages");

template <int NDP>
struct TmaTile {
    static constexpr uint32_t kGradBytes = kTile * 2;
    static constexpr uint32_t kStateBytes = kTile * 4;
    static constexpr uint32_t kStageBytes = NDP * kGradBytes + 3 * kStateBytes;
    static constexpr uint32_t kSmemBytes = kStages * kStageBytes;
};

template <int NDP>
__global__ void __launch_bounds__(kTmaThreads, 2)
rs_adamw_tma_kernel(const __grid_constant__ UpdateParams p, int64_t n_tiles) {
    using Tile = TmaTile<NDP>;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) uint64_t full[kStages];
    const int tid = threadIdx.x;
    const float coef = clip_coef(p.h);
    const StepScalars sc = step_scalars(p.h);
    const int64_t n8 = (p.n >> 3) << 3;                   // the tiles cover [0, n8)
    // the k-th tile of this CTA
#if ZGB_TMA_INTERLEAVE
    const int64_t count = blockIdx.x < n_tiles ? (n_tiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    auto tile_of = [&](int64_t k) { return (int64_t)blockIdx.x + k * gridDim.x; };
#else
    const int64_t per = (n_tiles + gridDim.x - 1) / gridDim.x;
    const int64_t t0 = (int64_t)blockIdx.x * per;
    const int64_t count = t0 < n_tiles ? min(per, n_tiles - t0) : 0;
    auto tile_of = [&](int64_t k) { return t0 + k; };
#endif

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&full[s], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    // thread 0 only: stage s <- tile t0 + k
    auto issue = [&](int64_t k, int s) {
        const int64_t e0 = tile_of(k) * kTile;
        const uint32_t elems = (uint32_t)min((int64_t)kTile, n8 - e0);   // a multiple of 8
        unsigned char* st = smem + (size_t)s * Tile::kStageBytes;
        mbar_arrive_expect_tx(&full[s], elems * (2u * NDP + 12u));
#pragma unroll
        for (int r = 0; r < NDP; ++r)
            bulk_g2s(st + r * Tile::kGradBytes, static_cast<const uint16_t*>(p.src[r]) + e0, elems * 2,
                     &full[s]);
        bulk_g2s(st + NDP * Tile::kGradBytes, p.w + e0, elems * 4, &full[s]);
        bulk_g2s(st + NDP * Tile::kGradBytes + Tile::kStateBytes, p.m + e0, elems * 4, &full[s]);
        bulk_g2s(st + NDP * Tile::kGradBytes + 2 * Tile::kStateBytes, p.v + e0, elems * 4, &full[s]);
    };

    if (tid == 0)
        for (int s = 0; s < kStages && s < count; ++s) issue(s, s);

    int64_t k = 0;
    bool ok = true;
    for (; k < count; ++k) {
        const int s = (int)(k % kStages);
        const uint32_t parity = (uint32_t)((k / kStages) & 1);
        ok = __syncthreads_and(mbar_wait_bounded(&full[s], parity, ZGB_TMA_TIMEOUT_CYCLES)) != 0;
        if (!ok) break;
        const int64_t e0 = tile_of(k) * kTile;
        const int64_t elems = min((int64_t)kTile, n8 - e0);
        const int j = tid * 4;
        if (j < elems) {
            const unsigned char* st = smem + (size_t)s * Tile::kStageBytes;
            float sum[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
            for (int r = 0; r < NDP; ++r) {
                const uint2 g = *reinterpret_cast<const uint2*>(st + r * Tile::kGradBytes + j * 2);
                sum[0] = __fadd_rn(sum[0], bf16_lo(g.x));
                sum[1] = __fadd_rn(sum[1], bf16_hi(g.x));
                sum[2] = __fadd_rn(sum[2], bf16_lo(g.y));
                sum[3] = __fadd_rn(sum[3], bf16_hi(g.y));
            }
            const unsigned char* sb = st + NDP * Tile::kGradBytes;
            const float4 w4 = *reinterpret_cast<const float4*>(sb + j * 4);
            const float4 m4 = *reinterpret_cast<const float4*>(sb + Tile::kStateBytes + j * 4);
            const float4 v4 = *reinterpret_cast<const float4*>(sb + 2 * Tile::kStateBytes + j * 4);
            float w[4] = {w4.x, w4.y, w4.z, w4.w};
            float m[4] = {m4.x, m4.y, m4.z, m4.w};
            float v[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) adamw_update(mean_grad(sum[q], p.h, coef), w[q], m[q], v[q], p.h, sc);
            st_stream_f4(p.w + e0 + j, make_float4(w[0], w[1], w[2], w[3]));
            st_stream_f4(p.m + e0 + j, make_float4(m[0], m[1], m[2], m[3]));
            st_stream_f4(p.v + e0 + j, make_float4(v[0], v[1], v[2], v[3]));
            *reinterpret_cast<uint2*>(p.out + e0 + j) =
                make_uint2(pack_bf16x2(w[0], w[1]), pack_bf16x2(w[2], w[3]));
        }
        __syncthreads();                                   // every thread is done with stage s
        if (tid == 0 && k + kStages < count) issue(k + kStages, s);
    }
    if (!ok) {
        // A wait gave up: record it, then wait (bounded) for the copies this
        // CTA still has in flight -- tiles k .. k + kStages - 1 -- and return.
        if (tid == 0) {
            atomicExch(&g_device_status, ZERO_ETIMEOUT);
            for (int64_t q = k; q < count && q < k + kStages; ++q)
                (void)mbar_wait_bounded(&full[q % kStages], (uint32_t)((q / kStages) & 1),
                                        ZGB_TMA_TIMEOUT_CYCLES);
        }
        __syncthreads();
        return;
    }
    // the last n % 8 elements, element by element, in CTA 0
    if (blockIdx.x == 0 && tid < p.n - n8) {
        const int64_t i = n8 + tid;
        float sum = 0.0f;
        for (int r = 0; r < NDP; ++r) sum = __fadd_rn(sum, bf16_one(static_cast<const uint16_t*>(p.src[r])[i]));
        float w = p.w[i], m = p.m[i], v = p.v[i];
        adamw_update(mean_grad(sum, p.h, coef), w, m, v, p.h, sc);
        p.w[i] = w;
        p.m[i] = m;
        p.v[i] = v;
        p.out[i] = to_bf16(w);
    }
}

template <int NDP>
int launch_tma(const UpdateParams& p, cudaStream_t stream) {
    using Tile = TmaTile<NDP>;
    // the opt-in above the default 48 KB of dynamic shared memory, per device:
    // set before every launch (cheap next to the launch) so that any thread and
    // any current device is covered
    const cudaError_t e = cudaFuncSetAttribute((const void*)rs_adamw_tma_kernel<NDP>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)Tile::kSmemBytes);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        note_cuda_error(e);
        return ZERO_ECUDA;
    }
    const int occupancy = ctas_per_sm((const void*)rs_adamw_tma_kernel<NDP>, kTmaThreads, Tile::kSmemBytes);
    const int64_t n_tiles = ((p.n >> 3) * 8 + kTile - 1) / kTile;
    const int64_t resident = (int64_t)sm_count() * occupancy;
    const unsigned grid = (unsigned)(n_tiles < 1 ? 1 : (n_tiles < resident ? n_tiles : resident));
    rs_adamw_tma_kernel<NDP><<<grid, kTmaThreads, Tile::kSmemBytes, stream>>>(p, n_tiles);
    return launch_status();
}

// ----------------------------------------------------------------------------
// Warp-specialized variant.  Warp 0 is the producer: its lane 0 issues the bulk
// copies of tile k into stage k % S once every consumer warp has released that
// stage's previous tile (an "empty" mbarrier with one arrival per consumer
// warp), and arms the stage's "full" mbarrier with the tile's byte count.
// Warps 1..C are consumers: each waits for the stage to be full, updates its
// 128 elements of the tile (4 per lane; tile = 128 C) from shared memory, stores the results
// to global memory, and arrives on the stage's empty barrier.  No barrier of
// the whole CTA sits inside the loop, so a slow warp delays only the refill of
// the one stage it still holds.  Tile u of a stage completes phase u of both
// barriers; waits pass the parity u & 1 (a wait never trails by two phases:
// the producer cannot refill before every consumer released, and a consumer
// cannot release a tile that was not issued).
//
// Bounded waits everywhere: a wait that gives up records ZERO_ETIMEOUT and
// ends that warp's loop.  The producer then waits, bounded again, for the
// copies of the last S issued tiles before it exits, so that no copy lands in
// the shared memory of a finished CTA.
constexpr int kWsConsumerWarps = ZGB_WS_CONSUMERS;
constexpr int kWsThreads = 32 * (kWsConsumerWarps + 1);
constexpr int kWsStages = ZGB_WS_STAGES;
constexpr int kWsTile = 4 * 32 * kWsConsumerWarps;       // a consumer lane updates 4 elements
static_assert(kWsStages >= 2 && kWsStages <= 8, "the warp-specialized ring runs with 2 to 8 stages");
static_assert(kWsConsumerWarps >= 1 && kWsConsumerWarps <= 31, "at most 32 warps per CTA");

template <int NDP>
struct WsTile {
    static constexpr uint32_t kGradBytes = kWsTile * 2;
    static constexpr uint32_t kStateBytes = kWsTile * 4;
    static constexpr uint32_t kStageBytes = NDP * kGradBytes + 3 * kStateBytes;
    static constexpr uint32_t kSmemBytes = kWsStages * kStageBytes;
};
static_assert(WsTile<8>::kSmemBytes <= 227 * 1024, "the ring must fit the shared memory of one CTA");

template <int NDP>
__global__ void __launch_bounds__(kWsThreads, 1)
rs_adamw_ws_kernel(const __grid_constant__ UpdateParams p, int64_t n_tiles) {
    using Tile = WsTile<NDP>;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) uint64_t full[kWsStages];
    __shared__ __align__(8) uint64_t empty[kWsStages];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t n8 = (p.n >> 3) << 3;
    const int64_t count = blockIdx.x < n_tiles ? (n_tiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    auto tile_e0 = [&](int64_t k) { return ((int64_t)blockIdx.x + k * gridDim.x) * kWsTile; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kWsStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kWsConsumerWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (warp == 0) {
        if (lane == 0) {
            int64_t k = 0;
            for (; k < count; ++k) {
                const int s = (int)(k % kWsStages);
                if (k >= kWsStages &&
                    !mbar_wait_bounded(&empty[s], (uint32_t)((k / kWsStages - 1) & 1), ZGB_TMA_TIMEOUT_CYCLES)) {
                    atomicExch(&g_device_status, ZERO_ETIMEOUT);
                    break;
                }
                const int64_t e0 = tile_e0(k);
                const uint32_t elems = (uint32_t)min((int64_t)kWsTile, n8 - e0);     // a multiple of 8
                unsigned char* st = smem + (size_t)s * Tile::kStageBytes;
                mbar_arrive_expect_tx(&full[s], elems * (2u * NDP + 12u));
#pragma unroll
                for (int r = 0; r < NDP; ++r)
                    bulk_g2s(st + r * Tile::kGradBytes, static_cast<const uint16_t*>(p.src[r]) + e0,
                             elems * 2, &full[s]);
                bulk_g2s(st + NDP * Tile::kGradBytes, p.w + e0, elems * 4, &full[s]);
                bulk_g2s(st + NDP * Tile::kGradBytes + Tile::kStateBytes, p.m + e0, elems * 4, &full[s]);
                bulk_g2s(st + NDP * Tile::kGradBytes + 2 * Tile::kStateBytes, p.v + e0, elems * 4, &full[s]);
            }
            // the copies of the last stages issued must land before the CTA ends
            for (int64_t j = k > kWsStages ? k - kWsStages : 0; j < k; ++j)
                (void)mbar_wait_bounded(&full[j % kWsStages], (uint32_t)((j / kWsStages) & 1),
                                        ZGB_TMA_TIMEOUT_CYCLES);
        }
    } else {
        const float coef = clip_coef(p.h);
        const StepScalars sc = step_scalars(p.h);
        const int j = (warp - 1) * 128 + lane * 4;
        for (int64_t k = 0; k < count; ++k) {
            const int s = (int)(k % kWsStages);
            const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full[s], (uint32_t)((k / kWsStages) & 1),
                                                                      ZGB_TMA_TIMEOUT_CYCLES));
            if (!ok) {
                if (lane == 0) atomicExch(&g_device_status, ZERO_ETIMEOUT);
                break;
            }
            const int64_t e0 = tile_e0(k);
            if (j < min((int64_t)kWsTile, n8 - e0)) {
                const unsigned char* st = smem + (size_t)s * Tile::kStageBytes;
                float sum[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                for (int r = 0; r < NDP; ++r) {
                    const uint2 g = *reinterpret_cast<const uint2*>(st + r * Tile::kGradBytes + j * 2);
                    sum[0] = __fadd_rn(sum[0], bf16_lo(g.x));
                    sum[1] = __fadd_rn(sum[1], bf16_hi(g.x));
                    sum[2] = __fadd_rn(sum[2], bf16_lo(g.y));
                    sum[3] = __fadd_rn(sum[3], bf16_hi(g.y));
                }
                const unsigned char* sb = st + NDP * Tile::kGradBytes;
                const float4 w4 = *reinterpret_cast<const float4*>(sb + j * 4);
                const float4 m4 = *reinterpret_cast<const float4*>(sb + Tile::kStateBytes + j * 4);
                const float4 v4 = *reinterpret_cast<const float4*>(sb + 2 * Tile::kStateBytes + j * 4);
                float w[4] = {w4.x, w4.y, w4.z, w4.w};
                float m[4] = {m4.x, m4.y, m4.z, m4.w};
                float v[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) adamw_update(mean_grad(sum[q], p.h, coef), w[q], m[q], v[q], p.h, sc);
                st_stream_f4(p.w + e0 + j, make_float4(w[0], w[1], w[2], w[3]));
                st_stream_f4(p.m + e0 + j, make_float4(m[0], m[1], m[2], m[3]));
                st_stream_f4(p.v + e0 + j, make_float4(v[0], v[1], v[2], v[3]));
                *reinterpret_cast<uint2*>(p.out + e0 + j) =
                    make_uint2(pack_bf16x2(w[0], w[1]), pack_bf16x2(w[2], w[3]));
            }
            __syncwarp();                                     // the warp is done with stage s
            if (lane == 0) mbar_arrive(&empty[s]);
        }
        // the last n % 8 elements, element by element, in CTA 0's first consumer warp
        if (blockIdx.x == 0 && warp == 1 && lane < p.n - n8) {
            const int64_t i = n8 + lane;
            float sum = 0.0f;
            for (int r = 0; r < NDP; ++r)
                sum = __fadd_rn(sum, bf16_one(static_cast<const uint16_t*>(p.src[r])[i]));
            float w = p.w[i], m = p.m[i], v = p.v[i];
            adamw_update(mean_grad(sum, p.h, coef), w, m, v, p.h, sc);
            p.w[i] = w;
            p.m[i] = m;
            p.v[i] = v;
            p.out[i] = to_bf16(w);
        }
    }
}

template <int NDP>
int launch_ws(const UpdateParams& p, cudaStream_t stream) {
    using Tile = WsTile<NDP>;
    const cudaError_t e = cudaFuncSetAttribute((const void*)rs_adamw_ws_kernel<NDP>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)Tile::kSmemBytes);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        note_cuda_error(e);
        return ZERO_ECUDA;
    }
    const int occupancy = ctas_per_sm((const void*)rs_adamw_ws_kernel<NDP>, kWsThreads, Tile::kSmemBytes);
    const int64_t n_tiles = ((p.n >> 3) * 8 + kWsTile - 1) / kWsTile;
    const int64_t resident = (int64_t)sm_count() * occupancy;
    const unsigned grid = (unsigned)(n_tiles < 1 ? 1 : (n_tiles < resident ? n_tiles : resident));
    rs_adamw_ws_kernel<NDP><<<grid, kWsThreads, Tile::kSmemBytes, stream>>>(p, n_tiles);
    return launch_status();
}

int launch_rs_adamw_tma(const UpdateParams& p, cudaStream_t stream) {
    switch (p.n_src) {
        case 1: return ZGB_TMA_WS ? launch_ws<1>(p, stream) : launch_tma<1>(p, stream);
        case 2: return ZGB_TMA_WS ? launch_ws<2>(p, stream) : launch_tma<2>(p, stream);
        case 4: return ZGB_TMA_WS ? launch_ws<4>(p, stream) : launch_tma<4>(p, stream);
        case 8: return ZGB_TMA_WS ? launch_ws<8>(p, stream) : launch_tma<8>(p, stream);
        default: return 1;   // not applicable: the caller uses the register-staged kernel
    }
}

// One CTA waits on an mbarrier that nothing completes, with a short bound:
// the wait must give up, record ZERO_ETIMEOUT and return.
__global__ void bounded_wait_selftest_kernel(long long limit) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const bool ok = __syncthreads_and(mbar_wait_bounded(&bar, 0, limit)) != 0;
    if (!ok && threadIdx.x == 0) atomicExch(&g_device_status, ZERO_ETIMEOUT);
}

int take_device_status() {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof v) != cudaSuccess) {
        (void)cudaGetLastError();
        return ZERO_ECUDA;
    }
    if (v != ZERO_OK) {
        const int zero = ZERO_OK;
        if (cudaMemcpyToSymbol(g_device_status, &zero, sizeof zero) != cudaSuccess) {
            (void)cudaGetLastError();
            return ZERO_ECUDA;
        }
    }
    return v == ZERO_OK ? ZERO_OK : ZERO_ETIMEOUT;
}

}  // namespace zgb

extern "C" int zero_selftest_bounded_wait(int64_t limit_cycles, void* stream) {
    if (limit_cycles < 1 || limit_cycles > (1ll << 32)) return ZERO_EINVAL;
    zgb::bounded_wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(limit_cycles);
    return zgb::launch_status();
}
