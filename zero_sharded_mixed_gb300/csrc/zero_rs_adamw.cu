// Fused reduce-scatter (mean) + AdamW + bf16 cast + all-gather write, sm_103a.
//
// What it computes is stated in zero_gb300.h (zero_reduce_scatter_adamw):
// "ZeRO and FSDP", section "The idea, one stage at a time" -- rank r receives
// the average over ranks of shard r of the gradients, updates its fp32 master
// shard with Adam (exercise "A sharded Adam step": bias correction at step t,
// eps outside the square root) plus decoupled weight decay, casts to bf16 and
// all-gathers.  The simulated ranks live in this GPU's memory, so one pass over
// the owned range does the whole step: each element's n_src gradient values
// are read once, its 12 bytes of fp32 state are read and written once and its
// bf16 weight is written once, (26 + 2*n_src) bytes for bf16 sources.
//
// Design: a bandwidth-bound stream.  Each thread owns 8 consecutive elements
// per iteration: one 128-bit load per bf16 source slice, two per fp32 state
// array, the same stores, and one 128-bit bf16 store; all loads of an iteration
// are issued before any arithmetic, so a warp keeps (2*n_src + 6) x 512 bytes
// in flight.  Loads and stores are evict-first (each byte is touched once).
// A grid-stride loop over 8-element vectors, with the grid sized to the CTAs
// that are resident at once, keeps the tail to at most one partial wave.
//
// Arithmetic: every fp32 operation is an explicit IEEE round-to-nearest
// intrinsic (__fadd_rn, __fmul_rn, __fdiv_rn, __fsqrt_rn), so nothing is fused
// into an FMA and the result is reproducible: the sum runs over ranks in
// ascending order from +0.0f, divides once, and the AdamW operations run in the
// order written in the header.
#include <cmath>

#include "zero_common.cuh"

#ifndef ZGB_RS_WAVES
#define ZGB_RS_WAVES 1       // grid = resident CTAs x this (grid-stride loop inside)
#endif
#ifndef ZGB_RS_MULTI
#define ZGB_RS_MULTI 1       // 0: one vector per thread and iteration everywhere
#endif
#ifndef ZGB_RS_MINBLOCKS
#define ZGB_RS_MINBLOCKS 1   // CTAs per SM the register allocation must allow
#endif

namespace zgb {

struct RsAdamwParams {
    const void* src[ZERO_MAX_SRC];  // already offset to the first element of the range
    float* w;
    float* m;
    float* v;
    uint16_t* out;
    int64_t n;                      // elements in the range
    int32_t n_src;
    float divisor;
    float b1, b2, omb1, omb2;       // beta1, beta2, 1-beta1, 1-beta2 (fp32)
    float bc1, bc2;                 // bias corrections 1-beta^t (fp64 -> fp32)
    float lr, lrwd, eps;            // lr, lr*wd (fp32), eps
};

__device__ __forceinline__ void adamw_update(float g, float& w, float& m, float& v,
                                             const RsAdamwParams& p) {
    const float mi = __fadd_rn(__fmul_rn(p.b1, m), __fmul_rn(p.omb1, g));
    const float vi = __fadd_rn(__fmul_rn(p.b2, v), __fmul_rn(p.omb2, __fmul_rn(g, g)));
    const float m_hat = __fdiv_rn(mi, p.bc1);
    const float v_hat = __fdiv_rn(vi, p.bc2);
    float wi = __fsub_rn(w, __fmul_rn(p.lrwd, w));                       // decoupled decay
    const float denom = __fadd_rn(__fsqrt_rn(v_hat), p.eps);
    wi = __fsub_rn(wi, __fmul_rn(p.lr, __fdiv_rn(m_hat, denom)));         // Adam step
    w = wi;
    m = mi;
    v = vi;
}

__device__ __forceinline__ void add_bf16x8(float (&s)[8], const uint4 x) {
    s[0] = __fadd_rn(s[0], bf16_lo(x.x));
    s[1] = __fadd_rn(s[1], bf16_hi(x.x));
    s[2] = __fadd_rn(s[2], bf16_lo(x.y));
    s[3] = __fadd_rn(s[3], bf16_hi(x.y));
    s[4] = __fadd_rn(s[4], bf16_lo(x.z));
    s[5] = __fadd_rn(s[5], bf16_hi(x.z));
    s[6] = __fadd_rn(s[6], bf16_lo(x.w));
    s[7] = __fadd_rn(s[7], bf16_hi(x.w));
}

__device__ __forceinline__ void add_f32x8(float (&s)[8], const float4 a, const float4 b) {
    s[0] = __fadd_rn(s[0], a.x);
    s[1] = __fadd_rn(s[1], a.y);
    s[2] = __fadd_rn(s[2], a.z);
    s[3] = __fadd_rn(s[3], a.w);
    s[4] = __fadd_rn(s[4], b.x);
    s[5] = __fadd_rn(s[5], b.y);
    s[6] = __fadd_rn(s[6], b.z);
    s[7] = __fadd_rn(s[7], b.w);
}

// One 8-element vector.  NDP > 0: that many sources, fully unrolled so every
// load is in flight before the first add; NDP == 0: p.n_src sources in a loop.
template <int NDP, bool kBf16>
__device__ __forceinline__ void step_vec(const RsAdamwParams& p, int64_t vi) {
    const int64_t e = vi * 8;
    float s[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) s[j] = 0.0f;
    if constexpr (NDP > 0) {
        if constexpr (kBf16) {
            uint4 raw[NDP];
#pragma unroll
            for (int r = 0; r < NDP; ++r)
                raw[r] = ld_stream_u4(static_cast<const uint16_t*>(p.src[r]) + e);
#pragma unroll
            for (int r = 0; r < NDP; ++r) add_bf16x8(s, raw[r]);
        } else {
            float4 lo[NDP], hi[NDP];
#pragma unroll
            for (int r = 0; r < NDP; ++r) {
                lo[r] = ld_stream_f4(static_cast<const float*>(p.src[r]) + e);
                hi[r] = ld_stream_f4(static_cast<const float*>(p.src[r]) + e + 4);
            }
#pragma unroll
            for (int r = 0; r < NDP; ++r) add_f32x8(s, lo[r], hi[r]);
        }
    } else {
        for (int r = 0; r < p.n_src; ++r) {
            if constexpr (kBf16) {
                add_bf16x8(s, ld_stream_u4(static_cast<const uint16_t*>(p.src[r]) + e));
            } else {
                const float* q = static_cast<const float*>(p.src[r]) + e;
                add_f32x8(s, ld_stream_f4(q), ld_stream_f4(q + 4));
            }
        }
    }
    const float4 w0 = ld_stream_f4(p.w + e), w1 = ld_stream_f4(p.w + e + 4);
    const float4 m0 = ld_stream_f4(p.m + e), m1 = ld_stream_f4(p.m + e + 4);
    const float4 v0 = ld_stream_f4(p.v + e), v1 = ld_stream_f4(p.v + e + 4);
    float w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
    float m[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
    float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
    for (int j = 0; j < 8; ++j) adamw_update(__fdiv_rn(s[j], p.divisor), w[j], m[j], v[j], p);
    st_stream_f4(p.w + e, make_float4(w[0], w[1], w[2], w[3]));
    st_stream_f4(p.w + e + 4, make_float4(w[4], w[5], w[6], w[7]));
    st_stream_f4(p.m + e, make_float4(m[0], m[1], m[2], m[3]));
    st_stream_f4(p.m + e + 4, make_float4(m[4], m[5], m[6], m[7]));
    st_stream_f4(p.v + e, make_float4(v[0], v[1], v[2], v[3]));
    st_stream_f4(p.v + e + 4, make_float4(v[4], v[5], v[6], v[7]));
    uint4 o;
    o.x = pack_bf16x2(w[0], w[1]);
    o.y = pack_bf16x2(w[2], w[3]);
    o.z = pack_bf16x2(w[4], w[5]);
    o.w = pack_bf16x2(w[6], w[7]);
    st_stream_u4(p.out + e, o);
}

// One element (ragged tails and pointers that are not 16-byte aligned).
template <bool kBf16>
__device__ __forceinline__ void step_one(const RsAdamwParams& p, int64_t i) {
    float s = 0.0f;
    for (int r = 0; r < p.n_src; ++r) {
        const float x = kBf16 ? bf16_one(static_cast<const uint16_t*>(p.src[r])[i])
                              : static_cast<const float*>(p.src[r])[i];
        s = __fadd_rn(s, x);
    }
    float w = p.w[i], m = p.m[i], v = p.v[i];
    adamw_update(__fdiv_rn(s, p.divisor), w, m, v, p);
    p.w[i] = w;
    p.m[i] = m;
    p.v[i] = v;
    p.out[i] = to_bf16(w);
}

// U vectors per thread and iteration (vectors vi0, vi0 + stride, ...): every
// load of all U vectors is issued before the first add, so a thread keeps
// U * (loads per vector) 128-bit loads in flight.  Used when one vector alone
// has few loads (one or two sources), where a single vector per thread leaves
// HBM short of bytes in flight.
template <int NDP, bool kBf16, int U>
__device__ __forceinline__ void step_vecs(const RsAdamwParams& p, int64_t vi0, int64_t stride,
                                          int64_t nv) {
    static_assert(NDP > 0, "the multi-vector step needs a compile-time source count");
    constexpr int kRaw = kBf16 ? NDP : 2 * NDP;   // 128-bit source loads per vector
    uint4 graw[U][kBf16 ? kRaw : 1];
    float4 fraw[U][kBf16 ? 1 : kRaw];
    float4 st[U][6];
    bool ok[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int64_t vi = vi0 + u * stride;
        ok[u] = vi < nv;
        if (ok[u]) {
            const int64_t e = vi * 8;
#pragma unroll
            for (int r = 0; r < NDP; ++r) {
                if constexpr (kBf16) {
                    graw[u][r] = ld_stream_u4(static_cast<const uint16_t*>(p.src[r]) + e);
                } else {
                    fraw[u][2 * r] = ld_stream_f4(static_cast<const float*>(p.src[r]) + e);
                    fraw[u][2 * r + 1] = ld_stream_f4(static_cast<const float*>(p.src[r]) + e + 4);
                }
            }
            st[u][0] = ld_stream_f4(p.w + e);
            st[u][1] = ld_stream_f4(p.w + e + 4);
            st[u][2] = ld_stream_f4(p.m + e);
            st[u][3] = ld_stream_f4(p.m + e + 4);
            st[u][4] = ld_stream_f4(p.v + e);
            st[u][5] = ld_stream_f4(p.v + e + 4);
        }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
        if (!ok[u]) continue;
        const int64_t e = (vi0 + u * stride) * 8;
        float s[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) s[j] = 0.0f;
#pragma unroll
        for (int r = 0; r < NDP; ++r) {
            if constexpr (kBf16) add_bf16x8(s, graw[u][r]);
            else add_f32x8(s, fraw[u][2 * r], fraw[u][2 * r + 1]);
        }
        float w[8] = {st[u][0].x, st[u][0].y, st[u][0].z, st[u][0].w,
                      st[u][1].x, st[u][1].y, st[u][1].z, st[u][1].w};
        float m[8] = {st[u][2].x, st[u][2].y, st[u][2].z, st[u][2].w,
                      st[u][3].x, st[u][3].y, st[u][3].z, st[u][3].w};
        float v[8] = {st[u][4].x, st[u][4].y, st[u][4].z, st[u][4].w,
                      st[u][5].x, st[u][5].y, st[u][5].z, st[u][5].w};
#pragma unroll
        for (int j = 0; j < 8; ++j) adamw_update(__fdiv_rn(s[j], p.divisor), w[j], m[j], v[j], p);
        st_stream_f4(p.w + e, make_float4(w[0], w[1], w[2], w[3]));
        st_stream_f4(p.w + e + 4, make_float4(w[4], w[5], w[6], w[7]));
        st_stream_f4(p.m + e, make_float4(m[0], m[1], m[2], m[3]));
        st_stream_f4(p.m + e + 4, make_float4(m[4], m[5], m[6], m[7]));
        st_stream_f4(p.v + e, make_float4(v[0], v[1], v[2], v[3]));
        st_stream_f4(p.v + e + 4, make_float4(v[4], v[5], v[6], v[7]));
        uint4 o;
        o.x = pack_bf16x2(w[0], w[1]);
        o.y = pack_bf16x2(w[2], w[3]);
        o.z = pack_bf16x2(w[4], w[5]);
        o.w = pack_bf16x2(w[6], w[7]);
        st_stream_u4(p.out + e, o);
    }
}

// Vectors per thread and iteration: two when one vector has at most 8 loads.
template <int NDP, bool kBf16>
__host__ __device__ constexpr int vectors_per_iter() {
    return ZGB_RS_MULTI && NDP > 0 && ((kBf16 ? NDP : 2 * NDP) + 6) <= 8 ? 2 : 1;
}

template <int NDP, bool kBf16>
__global__ void __launch_bounds__(kThreads, ZGB_RS_MINBLOCKS)
rs_adamw_vec_kernel(const __grid_constant__ RsAdamwParams p) {
    const int64_t nv = p.n >> 3;
    const int64_t tid = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    constexpr int U = vectors_per_iter<NDP, kBf16>();
    if constexpr (U > 1) {
        for (int64_t vi = tid; vi < nv; vi += U * stride) step_vecs<NDP, kBf16, U>(p, vi, stride, nv);
    } else {
        for (int64_t vi = tid; vi < nv; vi += stride) step_vec<NDP, kBf16>(p, vi);
    }
    const int64_t tail = p.n - (nv << 3);
    if (tid < tail) step_one<kBf16>(p, (nv << 3) + tid);
}

template <bool kBf16>
__global__ void __launch_bounds__(kThreads)
rs_adamw_scalar_kernel(const __grid_constant__ RsAdamwParams p) {
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < p.n; i += stride)
        step_one<kBf16>(p, i);
}

template <int NDP, bool kBf16>
int launch_vec(const RsAdamwParams& p, cudaStream_t stream) {
    static int occupancy = 0;
    if (occupancy == 0) occupancy = ctas_per_sm((const void*)rs_adamw_vec_kernel<NDP, kBf16>, kThreads, 0);
    const int64_t resident = (int64_t)sm_count() * occupancy * ZGB_RS_WAVES;
    const unsigned grid = grid_for(p.n >> 3, kThreads, resident);
    rs_adamw_vec_kernel<NDP, kBf16><<<grid, kThreads, 0, stream>>>(p);
    return launch_status();
}

template <bool kBf16>
int launch_scalar(const RsAdamwParams& p, cudaStream_t stream) {
    static int occupancy = 0;
    if (occupancy == 0) occupancy = ctas_per_sm((const void*)rs_adamw_scalar_kernel<kBf16>, kThreads, 0);
    const unsigned grid = grid_for(p.n, kThreads, (int64_t)sm_count() * occupancy);
    rs_adamw_scalar_kernel<kBf16><<<grid, kThreads, 0, stream>>>(p);
    return launch_status();
}

template <bool kBf16>
int dispatch_vec(const RsAdamwParams& p, cudaStream_t s) {
    switch (p.n_src) {
        case 1: return launch_vec<1, kBf16>(p, s);
        case 2: return launch_vec<2, kBf16>(p, s);
        case 3: return launch_vec<3, kBf16>(p, s);
        case 4: return launch_vec<4, kBf16>(p, s);
        case 5: return launch_vec<5, kBf16>(p, s);
        case 6: return launch_vec<6, kBf16>(p, s);
        case 7: return launch_vec<7, kBf16>(p, s);
        case 8: return launch_vec<8, kBf16>(p, s);
        case 16: return launch_vec<16, kBf16>(p, s);
        default: return launch_vec<0, kBf16>(p, s);
    }
}

bool finite(float x) { return std::isfinite(x); }

}  // namespace zgb

extern "C" int zero_reduce_scatter_adamw(const zero_layout_t* L, const void* const* src,
                                         int32_t n_src, int32_t src_dtype, int64_t src_base,
                                         float divisor, int32_t rank_begin, int32_t rank_end,
                                         int64_t begin, int64_t end, float* master, float* m,
                                         float* v, uint16_t* out_bf16, int32_t out_mode,
                                         const zero_adamw_t* hp, void* stream) {
    using namespace zgb;
    // ---- arguments that need no CUDA call
    if (!L || !src || !master || !m || !v || !out_bf16 || !hp) return ZERO_EINVAL;
    if (n_src < 1) return ZERO_EINVAL;
    if (n_src > ZERO_MAX_SRC) return ZERO_ERANGE;
    if (src_dtype != ZERO_BF16 && src_dtype != ZERO_F32) return ZERO_EINVAL;
    if (out_mode != ZERO_OUT_FULL && out_mode != ZERO_OUT_SHARD) return ZERO_EINVAL;
    if (L->n_dp < 1 || L->shard < 0 || L->padded_n != L->shard * (int64_t)L->n_dp)
        return ZERO_EINVAL;
    if (rank_begin < 0 || rank_end > L->n_dp || rank_begin >= rank_end) return ZERO_EINVAL;
    const int64_t own_lo = (int64_t)rank_begin * L->shard;
    const int64_t own_hi = (int64_t)rank_end * L->shard;
    if (begin < own_lo || end > own_hi || begin > end) return ZERO_EINVAL;
    if (src_base > begin) return ZERO_EINVAL;
    if (!(divisor > 0.0f) || !finite(divisor)) return ZERO_EINVAL;
    if (hp->step < 1 || !finite(hp->lr) || !finite(hp->eps) || !finite(hp->weight_decay) ||
        !(hp->beta1 >= 0.0f && hp->beta1 < 1.0f) || !(hp->beta2 >= 0.0f && hp->beta2 < 1.0f))
        return ZERO_EINVAL;
    for (int r = 0; r < n_src; ++r)
        if (!src[r]) return ZERO_EINVAL;
    const int esize = src_dtype == ZERO_BF16 ? 2 : 4;
    for (int r = 0; r < n_src; ++r)
        if (check_aligned(src[r], esize)) return ZERO_EALIGN;
    if (check_aligned(master, 4) || check_aligned(m, 4) || check_aligned(v, 4) ||
        check_aligned(out_bf16, 2))
        return ZERO_EALIGN;
    if (end == begin) return ZERO_OK;

    // ---- pointer kinds (device memory of the current device)
    for (int r = 0; r < n_src; ++r)
        if (check_device_ptr(src[r])) return ZERO_EINVAL;
    if (check_device_ptr(master) || check_device_ptr(m) || check_device_ptr(v) ||
        check_device_ptr(out_bf16))
        return ZERO_EINVAL;

    // ---- parameters
    RsAdamwParams p;
    const int64_t state_off = begin - own_lo;
    const int64_t out_off = out_mode == ZERO_OUT_FULL ? begin : state_off;
    const int64_t src_off = begin - src_base;
    bool vec = true;
    for (int r = 0; r < ZERO_MAX_SRC; ++r) p.src[r] = nullptr;
    for (int r = 0; r < n_src; ++r) {
        p.src[r] = static_cast<const char*>(src[r]) + src_off * esize;
        vec = vec && aligned16(p.src[r]);
    }
    p.w = master + state_off;
    p.m = m + state_off;
    p.v = v + state_off;
    p.out = out_bf16 + out_off;
    vec = vec && aligned16(p.w) && aligned16(p.m) && aligned16(p.v) && aligned16(p.out);
    p.n = end - begin;
    p.n_src = n_src;
    p.divisor = divisor;
    p.b1 = hp->beta1;
    p.b2 = hp->beta2;
    p.omb1 = 1.0f - hp->beta1;
    p.omb2 = 1.0f - hp->beta2;
    p.bc1 = (float)(1.0 - std::pow((double)hp->beta1, (double)hp->step));
    p.bc2 = (float)(1.0 - std::pow((double)hp->beta2, (double)hp->step));
    p.lr = hp->lr;
    p.lrwd = hp->lr * hp->weight_decay;
    p.eps = hp->eps;
    if (!(p.bc1 > 0.0f) || !(p.bc2 > 0.0f)) return ZERO_EINVAL;   // beta == 0 at t >= 1 is fine; guards underflow

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool bf16 = src_dtype == ZERO_BF16;
    if (vec) return bf16 ? dispatch_vec<true>(p, s) : dispatch_vec<false>(p, s);
    return bf16 ? launch_scalar<true>(p, s) : launch_scalar<false>(p, s);
}
