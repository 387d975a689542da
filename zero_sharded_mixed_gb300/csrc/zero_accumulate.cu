// Gradient accumulation and the stage-3 per-layer gradient reduce-scatter, sm_103a.
//
// "ZeRO and FSDP", section "The idea, one stage at a time", paragraph on
// gradient accumulation: with several micro-batches per step, stage 1 adds each
// micro-batch's full local gradient into a full buffer and communicates once
// (ZERO_ACC_LOCAL: one source, per simulated rank); stage 2 reduce-scatters
// after every micro-batch (ZERO_ACC_REDUCE: the owner adds the sum over ranks
// of its slice into an fp32 shard buffer).  The stage-3 layer gradient
// reduce-scatter ("DeepSpeed ZeRO", "Stage 3 step by step", step 4) is
// ZERO_ACC_REDUCE with first = 1.
//
// Streaming kernel, 8 elements per thread per iteration: 128-bit loads of every
// source (bf16 or fp32), 2 x 128-bit loads of dst unless first, 2 x 128-bit
// stores.  Bytes per element: esize*n_src + 4 (+4 when accumulating).  Sums are
// explicit IEEE fp32 adds in ascending source order.
#include "zero_common.cuh"

#ifndef ZGB_ACC_LOCAL_U
#define ZGB_ACC_LOCAL_U 2    // vectors per thread and iteration, LOCAL mode
#endif
#ifndef ZGB_ACC_WAVES
#define ZGB_ACC_WAVES 64     // grid = resident CTAs x this: CTAs run in order over contiguous
                             // chunks (measured: +22 % for LOCAL, +10 % for REDUCE over x1)
#endif
#ifndef ZGB_ACC_REDUCE_U
#define ZGB_ACC_REDUCE_U 4   // the same for REDUCE with at most 4 source loads per vector
#endif

namespace zgb {

struct AccParams {
    const void* src[ZERO_MAX_SRC];  // offset to the first element of the range
    float* dst;                     // offset to the first element of the range
    int64_t n;
    int32_t n_src;
    int32_t first;
};

// kLocal: x = the single source value as is.  Otherwise x = +0 + sum over sources.
template <int NDP, bool kBf16, bool kLocal>
__device__ __forceinline__ void acc_vec(const AccParams& p, int64_t vi) {
    const int64_t e = vi * 8;
    float x[8];
    if constexpr (kLocal) {
        if constexpr (kBf16) {
            const uint4 a = ld_stream_u4(static_cast<const uint16_t*>(p.src[0]) + e);
            x[0] = bf16_lo(a.x); x[1] = bf16_hi(a.x); x[2] = bf16_lo(a.y); x[3] = bf16_hi(a.y);
            x[4] = bf16_lo(a.z); x[5] = bf16_hi(a.z); x[6] = bf16_lo(a.w); x[7] = bf16_hi(a.w);
        } else {
            const float4 a = ld_stream_f4(static_cast<const float*>(p.src[0]) + e);
            const float4 b = ld_stream_f4(static_cast<const float*>(p.src[0]) + e + 4);
            x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
            x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) x[j] = 0.0f;
        constexpr int kUnroll = NDP > 0 ? NDP : 1;
        const int n_src = NDP > 0 ? NDP : p.n_src;
        if constexpr (kBf16) {
            uint4 raw[kUnroll];
            for (int r0 = 0; r0 < n_src; r0 += kUnroll) {
#pragma unroll
                for (int r = 0; r < kUnroll; ++r)
                    if (NDP > 0 || r0 + r < n_src)
                        raw[r] = ld_stream_u4(static_cast<const uint16_t*>(p.src[r0 + r]) + e);
#pragma unroll
                for (int r = 0; r < kUnroll; ++r) {
                    if (NDP > 0 || r0 + r < n_src) {
                        const uint4 a = raw[r];
                        x[0] = __fadd_rn(x[0], bf16_lo(a.x)); x[1] = __fadd_rn(x[1], bf16_hi(a.x));
                        x[2] = __fadd_rn(x[2], bf16_lo(a.y)); x[3] = __fadd_rn(x[3], bf16_hi(a.y));
                        x[4] = __fadd_rn(x[4], bf16_lo(a.z)); x[5] = __fadd_rn(x[5], bf16_hi(a.z));
                        x[6] = __fadd_rn(x[6], bf16_lo(a.w)); x[7] = __fadd_rn(x[7], bf16_hi(a.w));
                    }
                }
            }
        } else {
            for (int r = 0; r < n_src; ++r) {
                const float* q = static_cast<const float*>(p.src[r]) + e;
                const float4 a = ld_stream_f4(q), b = ld_stream_f4(q + 4);
                x[0] = __fadd_rn(x[0], a.x); x[1] = __fadd_rn(x[1], a.y);
                x[2] = __fadd_rn(x[2], a.z); x[3] = __fadd_rn(x[3], a.w);
                x[4] = __fadd_rn(x[4], b.x); x[5] = __fadd_rn(x[5], b.y);
                x[6] = __fadd_rn(x[6], b.z); x[7] = __fadd_rn(x[7], b.w);
            }
        }
    }
    if (!p.first) {
        const float4 a = ld_stream_f4(p.dst + e), b = ld_stream_f4(p.dst + e + 4);
        x[0] = __fadd_rn(a.x, x[0]); x[1] = __fadd_rn(a.y, x[1]);
        x[2] = __fadd_rn(a.z, x[2]); x[3] = __fadd_rn(a.w, x[3]);
        x[4] = __fadd_rn(b.x, x[4]); x[5] = __fadd_rn(b.y, x[5]);
        x[6] = __fadd_rn(b.z, x[6]); x[7] = __fadd_rn(b.w, x[7]);
    }
    st_stream_f4(p.dst + e, make_float4(x[0], x[1], x[2], x[3]));
    st_stream_f4(p.dst + e + 4, make_float4(x[4], x[5], x[6], x[7]));
}

// U vectors per thread and iteration (vi0, vi0 + stride, ...; the kernel
// passes stride = kThreads, so a CTA's vectors are consecutive), all loads
// issued before the first add: the accumulation kernels move few bytes per vector
// (LOCAL: one 16-byte source load plus the 32-byte dst), so one vector per
// thread leaves HBM short of bytes in flight.
template <int NDP, bool kBf16, bool kLocal, int U>
__device__ __forceinline__ void acc_vecs(const AccParams& p, int64_t vi0, int64_t stride, int64_t nv) {
    constexpr int R = kLocal ? 1 : NDP;
    static_assert(R > 0, "the multi-vector step needs a compile-time source count");
    constexpr int kRaw = kBf16 ? R : 2 * R;
    uint4 graw[U][kBf16 ? kRaw : 1];
    float4 fraw[U][kBf16 ? 1 : kRaw];
    float4 d[U][2];
    bool ok[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int64_t vi = vi0 + u * stride;
        ok[u] = vi < nv;
        if (ok[u]) {
            const int64_t e = vi * 8;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                if constexpr (kBf16) {
                    graw[u][r] = ld_stream_u4(static_cast<const uint16_t*>(p.src[r]) + e);
                } else {
                    fraw[u][2 * r] = ld_stream_f4(static_cast<const float*>(p.src[r]) + e);
                    fraw[u][2 * r + 1] = ld_stream_f4(static_cast<const float*>(p.src[r]) + e + 4);
                }
            }
            if (!p.first) {
                d[u][0] = ld_stream_f4(p.dst + e);
                d[u][1] = ld_stream_f4(p.dst + e + 4);
            }
        }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
        if (!ok[u]) continue;
        const int64_t e = (vi0 + u * stride) * 8;
        float x[8];
        if constexpr (kLocal) {
            if constexpr (kBf16) {
                const uint4 a = graw[u][0];
                x[0] = bf16_lo(a.x); x[1] = bf16_hi(a.x); x[2] = bf16_lo(a.y); x[3] = bf16_hi(a.y);
                x[4] = bf16_lo(a.z); x[5] = bf16_hi(a.z); x[6] = bf16_lo(a.w); x[7] = bf16_hi(a.w);
            } else {
                const float4 a = fraw[u][0], b = fraw[u][1];
                x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
                x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) x[j] = 0.0f;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                if constexpr (kBf16) {
                    const uint4 a = graw[u][r];
                    x[0] = __fadd_rn(x[0], bf16_lo(a.x)); x[1] = __fadd_rn(x[1], bf16_hi(a.x));
                    x[2] = __fadd_rn(x[2], bf16_lo(a.y)); x[3] = __fadd_rn(x[3], bf16_hi(a.y));
                    x[4] = __fadd_rn(x[4], bf16_lo(a.z)); x[5] = __fadd_rn(x[5], bf16_hi(a.z));
                    x[6] = __fadd_rn(x[6], bf16_lo(a.w)); x[7] = __fadd_rn(x[7], bf16_hi(a.w));
                } else {
                    const float4 a = fraw[u][2 * r], b = fraw[u][2 * r + 1];
                    x[0] = __fadd_rn(x[0], a.x); x[1] = __fadd_rn(x[1], a.y);
                    x[2] = __fadd_rn(x[2], a.z); x[3] = __fadd_rn(x[3], a.w);
                    x[4] = __fadd_rn(x[4], b.x); x[5] = __fadd_rn(x[5], b.y);
                    x[6] = __fadd_rn(x[6], b.z); x[7] = __fadd_rn(x[7], b.w);
                }
            }
        }
        if (!p.first) {
            const float4 a = d[u][0], b = d[u][1];
            x[0] = __fadd_rn(a.x, x[0]); x[1] = __fadd_rn(a.y, x[1]);
            x[2] = __fadd_rn(a.z, x[2]); x[3] = __fadd_rn(a.w, x[3]);
            x[4] = __fadd_rn(b.x, x[4]); x[5] = __fadd_rn(b.y, x[5]);
            x[6] = __fadd_rn(b.z, x[6]); x[7] = __fadd_rn(b.w, x[7]);
        }
        st_stream_f4(p.dst + e, make_float4(x[0], x[1], x[2], x[3]));
        st_stream_f4(p.dst + e + 4, make_float4(x[4], x[5], x[6], x[7]));
    }
}

// Vectors per thread and iteration, chosen by measurement on GB300 (GPT-2-XL
// shapes): LOCAL does best with two; REDUCE with four while a vector has at
// most four source loads, one beyond that (eight bf16 sources already keep
// ten loads per vector in flight).
template <int NDP, bool kBf16, bool kLocal>
__host__ __device__ constexpr int acc_vectors_per_iter() {
    return kLocal ? ZGB_ACC_LOCAL_U
         : (NDP > 0 && (kBf16 ? NDP : 2 * NDP) <= 4) ? ZGB_ACC_REDUCE_U : 1;
}

template <bool kBf16, bool kLocal>
__device__ __forceinline__ void acc_one(const AccParams& p, int64_t i) {
    float x;
    if (kLocal) {
        x = kBf16 ? bf16_one(static_cast<const uint16_t*>(p.src[0])[i])
                  : static_cast<const float*>(p.src[0])[i];
    } else {
        x = 0.0f;
        for (int r = 0; r < p.n_src; ++r)
            x = __fadd_rn(x, kBf16 ? bf16_one(static_cast<const uint16_t*>(p.src[r])[i])
                                   : static_cast<const float*>(p.src[r])[i]);
    }
    p.dst[i] = p.first ? x : __fadd_rn(p.dst[i], x);
}

template <int NDP, bool kBf16, bool kLocal>
__global__ void __launch_bounds__(kThreads) acc_vec_kernel(const __grid_constant__ AccParams p) {
    const int64_t nv = p.n >> 3;
    const int64_t tid = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    constexpr int U = acc_vectors_per_iter<NDP, kBf16, kLocal>();
    if constexpr (U > 1) {
        // U x kThreads consecutive vectors per CTA and pass (thread t: t, t + kThreads, ...)
        const int64_t chunk = (int64_t)U * kThreads;
        for (int64_t v0 = (int64_t)blockIdx.x * chunk + threadIdx.x; v0 < nv; v0 += (int64_t)gridDim.x * chunk)
            acc_vecs<NDP, kBf16, kLocal, U>(p, v0, kThreads, nv);
    } else {
        for (int64_t vi = tid; vi < nv; vi += stride) acc_vec<NDP, kBf16, kLocal>(p, vi);
    }
    const int64_t tail = p.n - (nv << 3);
    if (tid < tail) acc_one<kBf16, kLocal>(p, (nv << 3) + tid);
}

template <bool kBf16, bool kLocal>
__global__ void __launch_bounds__(kThreads) acc_scalar_kernel(const __grid_constant__ AccParams p) {
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < p.n; i += stride)
        acc_one<kBf16, kLocal>(p, i);
}

template <int NDP, bool kBf16, bool kLocal>
int launch_acc_vec(const AccParams& p, cudaStream_t s) {
    const int occupancy = ctas_per_sm((const void*)acc_vec_kernel<NDP, kBf16, kLocal>, kThreads, 0);
    const int64_t per_cta = (int64_t)acc_vectors_per_iter<NDP, kBf16, kLocal>() * kThreads;
    const unsigned grid = grid_for(p.n >> 3, per_cta, (int64_t)sm_count() * occupancy * ZGB_ACC_WAVES);
    acc_vec_kernel<NDP, kBf16, kLocal><<<grid, kThreads, 0, s>>>(p);
    return launch_status();
}

template <bool kBf16, bool kLocal>
int launch_acc_scalar(const AccParams& p, cudaStream_t s) {
    const int occupancy = ctas_per_sm((const void*)acc_scalar_kernel<kBf16, kLocal>, kThreads, 0);
    const unsigned grid = grid_for(p.n, kThreads, (int64_t)sm_count() * occupancy);
    acc_scalar_kernel<kBf16, kLocal><<<grid, kThreads, 0, s>>>(p);
    return launch_status();
}

template <bool kBf16>
int dispatch_reduce(const AccParams& p, cudaStream_t s) {
    switch (p.n_src) {
        case 1: return launch_acc_vec<1, kBf16, false>(p, s);
        case 2: return launch_acc_vec<2, kBf16, false>(p, s);
        case 4: return launch_acc_vec<4, kBf16, false>(p, s);
        case 8: return launch_acc_vec<8, kBf16, false>(p, s);
        default: return launch_acc_vec<0, kBf16, false>(p, s);
    }
}

}  // namespace zgb

extern "C" int zero_accumulate(const zero_layout_t* L, int32_t mode, const void* const* src,
                               int32_t n_src, int32_t src_dtype, int64_t src_base, float* dst,
                               int64_t dst_base, int64_t begin, int64_t end, int32_t first,
                               void* stream) {
    using namespace zgb;
    if (!L || !src || !dst) return ZERO_EINVAL;
    if (mode != ZERO_ACC_LOCAL && mode != ZERO_ACC_REDUCE) return ZERO_EINVAL;
    if (n_src < 1) return ZERO_EINVAL;
    if (n_src > ZERO_MAX_SRC) return ZERO_ERANGE;
    if (mode == ZERO_ACC_LOCAL && n_src != 1) return ZERO_EINVAL;
    if (src_dtype != ZERO_BF16 && src_dtype != ZERO_F32) return ZERO_EINVAL;
    if (!layout_shape_ok(L))
        return ZERO_EINVAL;
    if (begin < 0 || end > L->padded_n || begin > end) return ZERO_EINVAL;
    if (src_base > begin || dst_base > begin) return ZERO_EINVAL;
    for (int r = 0; r < n_src; ++r)
        if (!src[r]) return ZERO_EINVAL;
    const int esize = src_dtype == ZERO_BF16 ? 2 : 4;
    for (int r = 0; r < n_src; ++r)
        if (check_aligned(src[r], esize)) return ZERO_EALIGN;
    if (check_aligned(dst, 4)) return ZERO_EALIGN;
    if (end == begin) return ZERO_OK;
    for (int r = 0; r < n_src; ++r)
        if (check_device_ptr(src[r])) return ZERO_EINVAL;
    if (check_device_ptr(dst)) return ZERO_EINVAL;

    AccParams p;
    bool vec = true;
    for (int r = 0; r < ZERO_MAX_SRC; ++r) p.src[r] = nullptr;
    for (int r = 0; r < n_src; ++r) {
        p.src[r] = static_cast<const char*>(src[r]) + (begin - src_base) * esize;
        vec = vec && aligned16(p.src[r]);
    }
    p.dst = dst + (begin - dst_base);
    vec = vec && aligned16(p.dst);
    p.n = end - begin;
    p.n_src = n_src;
    p.first = first ? 1 : 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool bf16 = src_dtype == ZERO_BF16;
    const bool local = mode == ZERO_ACC_LOCAL;
    if (!vec) {
        if (local) return bf16 ? launch_acc_scalar<true, true>(p, s) : launch_acc_scalar<false, true>(p, s);
        return bf16 ? launch_acc_scalar<true, false>(p, s) : launch_acc_scalar<false, false>(p, s);
    }
    if (local) return bf16 ? launch_acc_vec<1, true, true>(p, s) : launch_acc_vec<1, false, true>(p, s);
    return bf16 ? dispatch_reduce<true>(p, s) : dispatch_reduce<false>(p, s);
}
