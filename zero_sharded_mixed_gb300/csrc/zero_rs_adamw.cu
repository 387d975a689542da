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
// The same kernel template serves four kinds of gradient source:
//   kPlainBf16 / kPlainF32  sum over n_src buffers (bf16 gradients, or fp32
//                           accumulators after gradient accumulation);
//   kAccLocal               the last micro-batch of stage-1 accumulation fused
//                           in: sum over ranks of (acc_r + g_r);
//   kAccReduce              the last micro-batch of stage-2 accumulation fused
//                           in: A + (sum over ranks of g_r).
// Both fused kinds perform exactly the additions of the unfused sequence
// (zero_accumulate, then the update), in the same order, so their results are
// bit-identical to it while skipping one fp32 write and re-read per element.
//
// The output is the bf16 weights, or (zero_reduce_scatter_adamw_q8, kQ8) the
// same weights in the 8-bit block format: a warp's 256 consecutive elements are
// one quantization block, quantized in the epilogue.
//
// Design: a bandwidth-bound stream.  Each thread owns 8 consecutive elements
// per vector: one 128-bit load per bf16 source, two per fp32 array, the same
// stores, and one 128-bit bf16 store.  All loads of an iteration are issued
// before any arithmetic; when a vector has few loads, a thread takes two
// vectors per iteration.  Loads and stores are evict-first.  The grid is a
// measured number of resident waves (rs_waves), each CTA over one contiguous
// chunk of vectors, the consecutive vectors of a chunk on consecutive lanes.
//
// Arithmetic: every fp32 operation is an explicit IEEE round-to-nearest
// intrinsic, so nothing is fused into an FMA: the sum runs over ranks in
// ascending order from +0.0f, divides once, and the AdamW operations run in
// the order written in the header (zero_update.cuh).
#include <cmath>

#include "zero_update.cuh"

#ifndef ZGB_RS_WAVES
#define ZGB_RS_WAVES 0       // grid = resident CTAs x this; 0 = the measured choice per kind
#endif
#ifndef ZGB_RS_WAVES_F32
#define ZGB_RS_WAVES_F32 32  // the same for fp32 sources alone, when ZGB_RS_WAVES is 0
#endif
#ifndef ZGB_RS_MULTI
#define ZGB_RS_MULTI 1       // 0: one vector per thread and iteration everywhere
#endif
#ifndef ZGB_RS_TMA
#define ZGB_RS_TMA 0         // 1: bf16 sources go through the TMA-staged kernel (zero_rs_adamw_tma.cu)
#endif
#ifndef ZGB_RS_MINBLOCKS
#define ZGB_RS_MINBLOCKS 2   // CTAs per SM the register allocation must allow (caps at 128)
#endif

namespace zgb {

enum SrcKind { kPlainBf16 = 0, kPlainF32 = 1, kAccLocal = 2, kAccReduce = 3 };

// Whether a kind's kernels apply a power-of-two divisor as a multiply (mean_grad).
template <int KIND>
__host__ __device__ constexpr bool kPow2Kind() {
    return KIND != kPlainF32;
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

// acc (8 fp32) + g (8 bf16), elementwise, into x
__device__ __forceinline__ void acc_plus_bf16x8(float (&x)[8], const float4 a, const float4 b,
                                                const uint4 g) {
    x[0] = __fadd_rn(a.x, bf16_lo(g.x));
    x[1] = __fadd_rn(a.y, bf16_hi(g.x));
    x[2] = __fadd_rn(a.z, bf16_lo(g.y));
    x[3] = __fadd_rn(a.w, bf16_hi(g.y));
    x[4] = __fadd_rn(b.x, bf16_lo(g.z));
    x[5] = __fadd_rn(b.y, bf16_hi(g.z));
    x[6] = __fadd_rn(b.z, bf16_lo(g.w));
    x[7] = __fadd_rn(b.w, bf16_hi(g.w));
}

// Registers holding one vector's gradient-source loads.  R = compile-time
// source count (> 0).
template <int KIND, int R>
struct SrcRegs {
    uint4 g[(KIND == kPlainF32) ? 1 : R];                      // bf16 gradients
    float4 f[(KIND == kPlainF32 || KIND == kAccLocal) ? 2 * R  // fp32 sources / accumulators
             : (KIND == kAccReduce ? 2 : 1)];
};

template <int KIND, int R>
__device__ __forceinline__ void load_src(const UpdateParams& p, int64_t e, SrcRegs<KIND, R>& s) {
#pragma unroll
    for (int r = 0; r < R; ++r) {
        if constexpr (KIND != kPlainF32)
            s.g[r] = ld_stream_u4(static_cast<const uint16_t*>(p.src[r]) + e);
        if constexpr (KIND == kPlainF32) {
            s.f[2 * r] = ld_stream_f4(static_cast<const float*>(p.src[r]) + e);
            s.f[2 * r + 1] = ld_stream_f4(static_cast<const float*>(p.src[r]) + e + 4);
        }
        if constexpr (KIND == kAccLocal) {
            s.f[2 * r] = ld_stream_f4(p.acc[r] + e);
            s.f[2 * r + 1] = ld_stream_f4(p.acc[r] + e + 4);
        }
    }
    if constexpr (KIND == kAccReduce) {
        s.f[0] = ld_stream_f4(p.acc[0] + e);
        s.f[1] = ld_stream_f4(p.acc[0] + e + 4);
    }
}

// The source sum of one vector, in the order of the unfused definition.
template <int KIND, int R>
__device__ __forceinline__ void sum_src(const SrcRegs<KIND, R>& s, float (&x)[8]) {
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = 0.0f;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        if constexpr (KIND == kPlainBf16 || KIND == kAccReduce) add_bf16x8(x, s.g[r]);
        if constexpr (KIND == kPlainF32) add_f32x8(x, s.f[2 * r], s.f[2 * r + 1]);
        if constexpr (KIND == kAccLocal) {
            float a[8];
            acc_plus_bf16x8(a, s.f[2 * r], s.f[2 * r + 1], s.g[r]);    // the rank's final acc
            add_f32x8(x, make_float4(a[0], a[1], a[2], a[3]), make_float4(a[4], a[5], a[6], a[7]));
        }
    }
    if constexpr (KIND == kAccReduce) {                                  // A + (sum over ranks)
        const float4 a = s.f[0], b = s.f[1];
        x[0] = __fadd_rn(a.x, x[0]); x[1] = __fadd_rn(a.y, x[1]);
        x[2] = __fadd_rn(a.z, x[2]); x[3] = __fadd_rn(a.w, x[3]);
        x[4] = __fadd_rn(b.x, x[4]); x[5] = __fadd_rn(b.y, x[5]);
        x[6] = __fadd_rn(b.z, x[6]); x[7] = __fadd_rn(b.w, x[7]);
    }
}

// The same source sum with a runtime source count, loads one source at a time.
template <int KIND>
__device__ __forceinline__ void sum_src_dyn(const UpdateParams& p, int64_t e, float (&x)[8]) {
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = 0.0f;
    for (int r = 0; r < p.n_src; ++r) {
        if constexpr (KIND == kPlainBf16 || KIND == kAccReduce) {
            add_bf16x8(x, ld_stream_u4(static_cast<const uint16_t*>(p.src[r]) + e));
        } else if constexpr (KIND == kPlainF32) {
            const float* q = static_cast<const float*>(p.src[r]) + e;
            add_f32x8(x, ld_stream_f4(q), ld_stream_f4(q + 4));
        } else {
            float a[8];
            acc_plus_bf16x8(a, ld_stream_f4(p.acc[r] + e), ld_stream_f4(p.acc[r] + e + 4),
                            ld_stream_u4(static_cast<const uint16_t*>(p.src[r]) + e));
            add_f32x8(x, make_float4(a[0], a[1], a[2], a[3]), make_float4(a[4], a[5], a[6], a[7]));
        }
    }
    if constexpr (KIND == kAccReduce) {
        const float4 a = ld_stream_f4(p.acc[0] + e), b = ld_stream_f4(p.acc[0] + e + 4);
        x[0] = __fadd_rn(a.x, x[0]); x[1] = __fadd_rn(a.y, x[1]);
        x[2] = __fadd_rn(a.z, x[2]); x[3] = __fadd_rn(a.w, x[3]);
        x[4] = __fadd_rn(b.x, x[4]); x[5] = __fadd_rn(b.y, x[5]);
        x[6] = __fadd_rn(b.z, x[6]); x[7] = __fadd_rn(b.w, x[7]);
    }
}

// U vectors (vi0, vi0 + stride, ...; the kernel passes stride = kThreads, so a
// CTA's vectors are consecutive) with a compile-time source count R: every
// load of all U vectors is issued before the first add.
template <int KIND, int R, int U, bool kQ8>
__device__ __forceinline__ void step_vecs(const UpdateParams& p, int64_t vi0, int64_t stride,
                                          int64_t nv, float coef, const StepScalars& sc) {
    SrcRegs<KIND, R> src[U];
    float4 st[U][6];
    bool ok[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int64_t vi = vi0 + u * stride;
        ok[u] = vi < nv;
        if (ok[u]) {
            load_src<KIND, R>(p, vi * 8, src[u]);
            load_state(p, vi * 8, st[u]);
        }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
        if (!ok[u]) continue;
        float s[8];
        sum_src<KIND, R>(src[u], s);
        if constexpr (kQ8)
            finish_vec_q8<kPow2Kind<KIND>()>(p, (vi0 + u * stride) * 8, s, st[u], coef, sc, p.q, p.qscale);
        else
            finish_vec<kPow2Kind<KIND>()>(p, (vi0 + u * stride) * 8, s, st[u], coef, sc);
    }
}

// One vector with a runtime source count.
template <int KIND, bool kQ8>
__device__ __forceinline__ void step_vec_dyn(const UpdateParams& p, int64_t vi, float coef,
                                             const StepScalars& sc) {
    const int64_t e = vi * 8;
    float s[8];
    sum_src_dyn<KIND>(p, e, s);
    float4 st[6];
    load_state(p, e, st);
    if constexpr (kQ8)
        finish_vec_q8<kPow2Kind<KIND>()>(p, e, s, st, coef, sc, p.q, p.qscale);
    else
        finish_vec<kPow2Kind<KIND>()>(p, e, s, st, coef, sc);
}

// One element (ragged tails and ranges not on 16-byte boundaries).
template <int KIND>
__device__ __forceinline__ void step_one(const UpdateParams& p, int64_t i, float coef,
                                         const StepScalars& sc) {
    float s = 0.0f;
    for (int r = 0; r < p.n_src; ++r) {
        float x;
        if constexpr (KIND == kPlainF32) {
            x = static_cast<const float*>(p.src[r])[i];
        } else {
            x = bf16_one(static_cast<const uint16_t*>(p.src[r])[i]);
            if constexpr (KIND == kAccLocal) x = __fadd_rn(p.acc[r][i], x);
        }
        s = __fadd_rn(s, x);
    }
    if constexpr (KIND == kAccReduce) s = __fadd_rn(p.acc[0][i], s);
    float w = p.w[i], m = p.m[i], v = p.v[i];
    adamw_update(mean_grad(s, p.h, coef), w, m, v, p.h, sc);
    p.w[i] = w;
    p.m[i] = m;
    p.v[i] = v;
    p.out[i] = to_bf16(w);
}

// 128-bit loads per vector of one source kind (gradient sources plus state).
template <int KIND, int R>
__host__ __device__ constexpr int loads_per_vec() {
    return (KIND == kPlainBf16 ? R : KIND == kPlainF32 ? 2 * R : KIND == kAccLocal ? 3 * R : R + 2) + 6;
}

// Vectors per thread and iteration: two when one vector has at most 8 loads.
template <int KIND, int R>
__host__ __device__ constexpr int vectors_per_iter() {
    return ZGB_RS_MULTI && R > 0 && loads_per_vec<KIND, R>() <= 8 ? 2 : 1;
}

// Grid size in resident waves.  Oversubscribing the grid (CTAs run in launch
// order, each over its own contiguous chunk) keeps the active CTAs on one
// stretch of each stream, which DRAM serves better than a persistent grid
// whose every pass spans the whole range.  Measured on GB300 (GPT-2-XL and
// Llama-7B shapes): x64 for bf16 sources and the stage-1 fused finish, x8 for
// the stage-2 fused finish, x32 for fp32 sources (the ZeRO-3 unit update:
// +3.5 % over x1, x64 and x128 0.8 % and 3 % below x32).
template <int KIND, int R>
__host__ __device__ constexpr int rs_waves() {
    return ZGB_RS_WAVES > 0 ? ZGB_RS_WAVES
         : KIND == kPlainF32 ? ZGB_RS_WAVES_F32 : KIND == kAccReduce ? 8 : 64;
}

// kQ8: the output is 8-bit codes and block scales (p.q, p.qscale) instead of
// bf16; the host guarantees whole 256-element blocks (no tail).
template <int KIND, int R, bool kQ8 = false>
__global__ void __launch_bounds__(kThreads, ZGB_RS_MINBLOCKS)
rs_adamw_vec_kernel(const __grid_constant__ UpdateParams p) {
    const float coef = clip_coef(p.h);
    const StepScalars sc = step_scalars(p.h);
    const int64_t nv = p.n >> 3;
    const int64_t tid = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    if constexpr (R > 0) {
        // a CTA takes U x kThreads consecutive vectors per pass (thread t: t,
        // t + kThreads, ...), so the CTAs resident at any moment cover one
        // contiguous stretch of every stream
        constexpr int U = vectors_per_iter<KIND, R>();
        const int64_t chunk = (int64_t)U * kThreads;
        for (int64_t v0 = (int64_t)blockIdx.x * chunk + threadIdx.x; v0 < nv; v0 += (int64_t)gridDim.x * chunk)
            step_vecs<KIND, R, U, kQ8>(p, v0, kThreads, nv, coef, sc);
    } else {
        for (int64_t vi = tid; vi < nv; vi += stride) step_vec_dyn<KIND, kQ8>(p, vi, coef, sc);
    }
    if constexpr (!kQ8) {
        const int64_t tail = p.n - (nv << 3);
        if (tid < tail) step_one<KIND>(p, (nv << 3) + tid, coef, sc);
    }
}

template <int KIND>
__global__ void __launch_bounds__(kThreads) rs_adamw_scalar_kernel(const __grid_constant__ UpdateParams p) {
    const float coef = clip_coef(p.h);
    const StepScalars sc = step_scalars(p.h);
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < p.n; i += stride)
        step_one<KIND>(p, i, coef, sc);
}

template <int KIND, int R, bool kQ8 = false>
int launch_vec(const UpdateParams& p, cudaStream_t stream) {
    const int occupancy = ctas_per_sm((const void*)rs_adamw_vec_kernel<KIND, R, kQ8>, kThreads, 0);
    const int64_t resident = (int64_t)sm_count() * occupancy * rs_waves<KIND, R>();
    const int64_t per_cta = (R > 0 ? vectors_per_iter<KIND, R>() : 1) * (int64_t)kThreads;
    const unsigned grid = grid_for(p.n >> 3, per_cta, resident);
    rs_adamw_vec_kernel<KIND, R, kQ8><<<grid, kThreads, 0, stream>>>(p);
    return launch_status();
}

// The 8-bit-output kernels (vector path only): the source counts of the
// stage-3 workloads (1: the fp32 buffer; 8: the ranks' bf16 gradients) and a
// few more, the rest through the runtime-count kernel.
template <int KIND>
int dispatch_q8(const UpdateParams& p, cudaStream_t s) {
    switch (p.n_src) {
        case 1: return launch_vec<KIND, 1, true>(p, s);
        case 2: return launch_vec<KIND, 2, true>(p, s);
        case 4: return launch_vec<KIND, 4, true>(p, s);
        case 8: return launch_vec<KIND, 8, true>(p, s);
        default: return launch_vec<KIND, 0, true>(p, s);
    }
}

template <int KIND>
int launch_scalar(const UpdateParams& p, cudaStream_t stream) {
    const int occupancy = ctas_per_sm((const void*)rs_adamw_scalar_kernel<KIND>, kThreads, 0);
    const unsigned grid = grid_for(p.n, kThreads, (int64_t)sm_count() * occupancy);
    rs_adamw_scalar_kernel<KIND><<<grid, kThreads, 0, stream>>>(p);
    return launch_status();
}

template <int KIND>
int dispatch(const UpdateParams& p, bool vec, cudaStream_t s) {
    if (!vec) return launch_scalar<KIND>(p, s);
    if constexpr (KIND == kPlainBf16 && ZGB_RS_TMA) {
        const int rc = launch_rs_adamw_tma(p, s);
        if (rc <= 0) return rc;                           // > 0: not applicable here
    }
    if constexpr (KIND == kPlainBf16 || KIND == kPlainF32) {
        switch (p.n_src) {
            case 1: return launch_vec<KIND, 1>(p, s);
            case 2: return launch_vec<KIND, 2>(p, s);
            case 3: return launch_vec<KIND, 3>(p, s);
            case 4: return launch_vec<KIND, 4>(p, s);
            case 5: return launch_vec<KIND, 5>(p, s);
            case 6: return launch_vec<KIND, 6>(p, s);
            case 7: return launch_vec<KIND, 7>(p, s);
            case 8: return launch_vec<KIND, 8>(p, s);
            case 16: return launch_vec<KIND, 16>(p, s);
            default: return launch_vec<KIND, 0>(p, s);
        }
    } else {
        switch (p.n_src) {
            case 1: return launch_vec<KIND, 1>(p, s);
            case 2: return launch_vec<KIND, 2>(p, s);
            case 4: return launch_vec<KIND, 4>(p, s);
            case 8: return launch_vec<KIND, 8>(p, s);
            default: return launch_vec<KIND, 0>(p, s);
        }
    }
}

// ----------------------------------------------------------------- host checks

int prepare_target(const zero_layout_t* L, int32_t rank_begin, int32_t rank_end, int64_t begin,
                   int64_t end, float* master, float* m, float* v, uint16_t* out, int32_t out_mode,
                   bool q8_out, UpdateTarget* t) {
    if (!L || !master || !m || !v) return ZERO_EINVAL;
    if (q8_out) {
        if (out_mode != ZERO_OUT_NONE || out != nullptr) return ZERO_EINVAL;
    } else if ((out_mode != ZERO_OUT_FULL && out_mode != ZERO_OUT_SHARD) || out == nullptr) {
        return ZERO_EINVAL;
    }
    if (!layout_shape_ok(L)) return ZERO_EINVAL;
    if (rank_begin < 0 || rank_end > L->n_dp || rank_begin >= rank_end) return ZERO_EINVAL;
    const int64_t own_lo = (int64_t)rank_begin * L->shard;
    const int64_t own_hi = (int64_t)rank_end * L->shard;
    if (begin < own_lo || end > own_hi || begin > end) return ZERO_EINVAL;
    if (check_aligned(master, 4) || check_aligned(m, 4) || check_aligned(v, 4) ||
        (out && check_aligned(out, 2)))
        return ZERO_EALIGN;
    const int64_t state_off = begin - own_lo;
    t->w = master + state_off;
    t->m = m + state_off;
    t->v = v + state_off;
    t->out = out ? out + (out_mode == ZERO_OUT_FULL ? begin : state_off) : nullptr;
    t->n = end - begin;
    t->aligned = aligned16(t->w) && aligned16(t->m) && aligned16(t->v) && (!t->out || aligned16(t->out));
    return ZERO_OK;
}

int check_target_ptrs(const UpdateTarget& t) {
    if (check_device_ptr(t.w) || check_device_ptr(t.m) || check_device_ptr(t.v) ||
        (t.out && check_device_ptr(t.out)))
        return ZERO_EINVAL;
    return ZERO_OK;
}

void bias_corrections(float b1, float b2, int64_t t, float* bc1, float* bc2) {
    *bc1 = (float)(1.0 - std::pow((double)b1, (double)t));
    *bc2 = (float)(1.0 - std::pow((double)b2, (double)t));
}

int make_scalars(const zero_adamw_t* hp, float divisor, AdamwScalars* h) {
    if (!hp) return ZERO_EINVAL;
    if (!(divisor > 0.0f) || !std::isfinite(divisor)) return ZERO_EINVAL;
    if (!std::isfinite(hp->eps) || !std::isfinite(hp->weight_decay) ||
        !(hp->beta1 >= 0.0f && hp->beta1 < 1.0f) || !(hp->beta2 >= 0.0f && hp->beta2 < 1.0f))
        return ZERO_EINVAL;
    h->divisor = divisor;
    int e2 = 0;
    const float mant = std::frexp(divisor, &e2);          // divisor = mant * 2^e2, mant in [0.5, 1)
    h->inv_divisor = (mant == 0.5f && e2 >= -125 && e2 <= 127) ? std::ldexp(1.0f, 1 - e2) : 0.0f;
    h->b1 = hp->beta1;
    h->b2 = hp->beta2;
    h->omb1 = 1.0f - hp->beta1;
    h->omb2 = 1.0f - hp->beta2;
    h->eps = hp->eps;
    h->wd = hp->weight_decay;
    h->max_norm = 0.0f;
    h->norm_sq = nullptr;
    h->sched = hp->sched;
    if (hp->sched) {                        // lr and the bias corrections come from the device
        if (check_aligned(hp->sched, 4)) return ZERO_EALIGN;
        if (check_device_ptr(hp->sched)) return ZERO_EINVAL;
        h->lr = h->lrwd = 0.0f;
        h->bc1 = h->bc2 = 1.0f;
        return ZERO_OK;
    }
    if (hp->step < 1 || !std::isfinite(hp->lr)) return ZERO_EINVAL;
    bias_corrections(hp->beta1, hp->beta2, hp->step, &h->bc1, &h->bc2);
    h->lr = hp->lr;
    h->lrwd = hp->lr * hp->weight_decay;
    if (!(h->bc1 > 0.0f) || !(h->bc2 > 0.0f)) return ZERO_EINVAL;
    return ZERO_OK;
}

// Shared body of the plain-source entry points (optionally clipped).
// q8 (optional): the 8-bit output -- codes laid out like the state and one
// scale per 256 elements of it -- in place of out (out_mode ZERO_OUT_NONE).
struct Q8Out {
    int8_t* q;
    float* scales;
};

int rs_adamw_plain(const zero_layout_t* L, const void* const* src, int32_t n_src, int32_t src_dtype,
                   int64_t src_base, float divisor, int32_t rank_begin, int32_t rank_end,
                   int64_t begin, int64_t end, float* master, float* m, float* v, uint16_t* out,
                   int32_t out_mode, const zero_adamw_t* hp, const double* norm_sq, float max_norm,
                   void* stream, const Q8Out* q8 = nullptr) {
    if (!src) return ZERO_EINVAL;
    if (n_src < 1) return ZERO_EINVAL;
    if (n_src > ZERO_MAX_SRC) return ZERO_ERANGE;
    if (src_dtype != ZERO_BF16 && src_dtype != ZERO_F32) return ZERO_EINVAL;
    UpdateTarget t;
    int rc = prepare_target(L, rank_begin, rank_end, begin, end, master, m, v, out, out_mode,
                            q8 != nullptr, &t);
    if (rc) return rc;
    if (src_base > begin) return ZERO_EINVAL;
    UpdateParams p;
    if ((rc = make_scalars(hp, divisor, &p.h))) return rc;
    if (norm_sq) {
        if (!(max_norm > 0.0f) || !std::isfinite(max_norm)) return ZERO_EINVAL;
        if (check_aligned(norm_sq, 8)) return ZERO_EALIGN;
        p.h.norm_sq = norm_sq;
        p.h.max_norm = max_norm;
    }
    for (int r = 0; r < n_src; ++r)
        if (!src[r]) return ZERO_EINVAL;
    const int esize = src_dtype == ZERO_BF16 ? 2 : 4;
    for (int r = 0; r < n_src; ++r)
        if (check_aligned(src[r], esize)) return ZERO_EALIGN;
    if (end == begin) return ZERO_OK;
    for (int r = 0; r < n_src; ++r)
        if (check_source_ptr(src[r])) return ZERO_EINVAL;
    if ((rc = check_target_ptrs(t))) return rc;
    if (norm_sq && check_device_ptr(norm_sq)) return ZERO_EINVAL;

    bool vec = t.aligned;
    for (int r = 0; r < ZERO_MAX_SRC; ++r) {
        p.src[r] = nullptr;
        p.acc[r] = nullptr;
    }
    for (int r = 0; r < n_src; ++r) {
        p.src[r] = static_cast<const char*>(src[r]) + (begin - src_base) * esize;
        vec = vec && aligned16(p.src[r]);
    }
    p.w = t.w;
    p.m = t.m;
    p.v = t.v;
    p.out = t.out;
    p.q = nullptr;
    p.qscale = nullptr;
    p.n = t.n;
    p.n_src = n_src;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (q8) {
        const int64_t state_off = begin - (int64_t)rank_begin * L->shard;   // a multiple of 256
        p.q = q8->q + state_off;
        p.qscale = q8->scales + state_off / 256;
        if (!vec || !aligned16(p.q)) return ZERO_EALIGN;
        return src_dtype == ZERO_BF16 ? dispatch_q8<kPlainBf16>(p, s) : dispatch_q8<kPlainF32>(p, s);
    }
    return src_dtype == ZERO_BF16 ? dispatch<kPlainBf16>(p, vec, s) : dispatch<kPlainF32>(p, vec, s);
}

}  // namespace zgb

extern "C" int zero_reduce_scatter_adamw(const zero_layout_t* L, const void* const* src,
                                         int32_t n_src, int32_t src_dtype, int64_t src_base,
                                         float divisor, int32_t rank_begin, int32_t rank_end,
                                         int64_t begin, int64_t end, float* master, float* m,
                                         float* v, uint16_t* out_bf16, int32_t out_mode,
                                         const zero_adamw_t* hp, void* stream) {
    return zgb::rs_adamw_plain(L, src, n_src, src_dtype, src_base, divisor, rank_begin, rank_end,
                               begin, end, master, m, v, out_bf16, out_mode, hp, nullptr, 0.0f,
                               stream);
}

extern "C" int zero_reduce_scatter_adamw_clip(const zero_layout_t* L, const void* const* src,
                                              int32_t n_src, int32_t src_dtype, int64_t src_base,
                                              float divisor, int32_t rank_begin, int32_t rank_end,
                                              int64_t begin, int64_t end, float* master, float* m,
                                              float* v, uint16_t* out_bf16, int32_t out_mode,
                                              const zero_adamw_t* hp, const double* norm_sq,
                                              float max_norm, void* stream) {
    if (!norm_sq) return ZERO_EINVAL;
    return zgb::rs_adamw_plain(L, src, n_src, src_dtype, src_base, divisor, rank_begin, rank_end,
                               begin, end, master, m, v, out_bf16, out_mode, hp, norm_sq, max_norm,
                               stream);
}

extern "C" int zero_reduce_scatter_adamw_q8(const zero_layout_t* L, const void* const* src,
                                            int32_t n_src, int32_t src_dtype, int64_t src_base,
                                            float divisor, int32_t rank_begin, int32_t rank_end,
                                            int64_t begin, int64_t end, float* master, float* m,
                                            float* v, int8_t* q_out, float* scales_out, int32_t block,
                                            const zero_adamw_t* hp, void* stream) {
    using namespace zgb;
    if (!L || !q_out || !scales_out) return ZERO_EINVAL;
    if (block != 256) return ZERO_EINVAL;
    if (L->shard % 256 != 0 || begin % 256 != 0 || end % 256 != 0) return ZERO_EINVAL;
    if (check_aligned(scales_out, 4)) return ZERO_EALIGN;
    if (end > begin && (check_device_ptr(q_out) || check_device_ptr(scales_out))) return ZERO_EINVAL;
    const Q8Out q8{q_out, scales_out};
    return rs_adamw_plain(L, src, n_src, src_dtype, src_base, divisor, rank_begin, rank_end, begin,
                          end, master, m, v, nullptr, ZERO_OUT_NONE, hp, nullptr, 0.0f, stream, &q8);
}

extern "C" int zero_accumulate_adamw(const zero_layout_t* L, int32_t mode,
                                     const float* const* acc, int32_t n_acc, int64_t acc_base,
                                     const uint16_t* const* grads, int32_t n_grads, int64_t grad_base,
                                     float divisor, int32_t rank_begin, int32_t rank_end,
                                     int64_t begin, int64_t end, float* master, float* m, float* v,
                                     uint16_t* out_bf16, int32_t out_mode, const zero_adamw_t* hp,
                                     void* stream) {
    using namespace zgb;
    if (!acc || !grads) return ZERO_EINVAL;
    if (mode != ZERO_ACC_LOCAL && mode != ZERO_ACC_REDUCE) return ZERO_EINVAL;
    if (n_grads < 1) return ZERO_EINVAL;
    if (n_grads > ZERO_MAX_SRC) return ZERO_ERANGE;
    if (mode == ZERO_ACC_LOCAL ? n_acc != n_grads : n_acc != 1) return ZERO_EINVAL;
    UpdateTarget t;
    int rc = prepare_target(L, rank_begin, rank_end, begin, end, master, m, v, out_bf16, out_mode,
                            false, &t);
    if (rc) return rc;
    if (acc_base > begin || grad_base > begin) return ZERO_EINVAL;
    UpdateParams p;
    if ((rc = make_scalars(hp, divisor, &p.h))) return rc;
    for (int r = 0; r < n_acc; ++r)
        if (!acc[r]) return ZERO_EINVAL;
    for (int r = 0; r < n_grads; ++r)
        if (!grads[r]) return ZERO_EINVAL;
    for (int r = 0; r < n_acc; ++r)
        if (check_aligned(acc[r], 4)) return ZERO_EALIGN;
    for (int r = 0; r < n_grads; ++r)
        if (check_aligned(grads[r], 2)) return ZERO_EALIGN;
    if (end == begin) return ZERO_OK;
    for (int r = 0; r < n_acc; ++r)
        if (check_device_ptr(acc[r])) return ZERO_EINVAL;
    for (int r = 0; r < n_grads; ++r)
        if (check_device_ptr(grads[r])) return ZERO_EINVAL;
    if ((rc = check_target_ptrs(t))) return rc;

    bool vec = t.aligned;
    for (int r = 0; r < ZERO_MAX_SRC; ++r) {
        p.src[r] = nullptr;
        p.acc[r] = nullptr;
    }
    for (int r = 0; r < n_grads; ++r) {
        p.src[r] = grads[r] + (begin - grad_base);
        vec = vec && aligned16(p.src[r]);
    }
    for (int r = 0; r < n_acc; ++r) {
        p.acc[r] = acc[r] + (begin - acc_base);
        vec = vec && aligned16(p.acc[r]);
    }
    p.w = t.w;
    p.m = t.m;
    p.v = t.v;
    p.out = t.out;
    p.q = nullptr;
    p.qscale = nullptr;
    p.n = t.n;
    p.n_src = n_grads;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return mode == ZERO_ACC_LOCAL ? dispatch<kAccLocal>(p, vec, s) : dispatch<kAccReduce>(p, vec, s);
}
