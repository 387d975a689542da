// The AdamW element update shared by every fused update kernel, and the host
// checks that place an update range on the owners' state.
//
// AdamW ("ZeRO and FSDP", exercise "A sharded Adam step": bias correction at
// step t, eps outside the square root; decoupled weight decay per the "AdamW"
// optimizer blocks of "DeepSpeed ZeRO", "The configuration file"):
//   m = b1*m + (1-b1)*g;  v = b2*v + (1-b2)*g*g;  mh = m/bc1;  vh = v/bc2;
//   w = w - (lr*wd)*w;    w = w - lr*(mh/(sqrt(vh)+eps))
// every operation one IEEE fp32 rounding (explicit _rn intrinsics, no FMA).
//
// Optional clipping by the global gradient norm ("DeepSpeed ZeRO", "The
// configuration file": gradient_clipping 1.0): with ||g||^2 in device memory,
// coef = min(1, fp32(max_norm / (sqrt(||g||^2) + 1e-6))) evaluated in fp64 and
// rounded once, and g is multiplied by coef before the update.
#pragma once

#include "zero_quant.cuh"

#ifndef ZGB_POW2_DIV
#define ZGB_POW2_DIV 1   // 1: the kernels that measured faster with it apply a power-of-two
                         // divisor as a multiply by its exact reciprocal (bit-identical)
#endif

namespace zgb {

struct AdamwScalars {
    float divisor;                  // g = sum / divisor
    float inv_divisor;              // 1 / divisor when that is an exact power of two, else 0
    float b1, b2, omb1, omb2;       // beta1, beta2, 1-beta1, 1-beta2 (fp32)
    float bc1, bc2;                 // 1 - beta^t in fp64, rounded to fp32
    float lr, lrwd, eps;            // lr, lr*wd (fp32), eps
    float wd;                       // weight decay (lr*wd is formed from it when sched is set)
    float max_norm;                 // clipping threshold (used when norm_sq is set)
    const double* norm_sq;          // device: squared global gradient norm, or nullptr
    const float* sched;             // device: {lr, bc1, bc2} of this step, or nullptr
};

// The scalars that change from step to step: from the parameters, or from
// device memory (zero_schedule_advance) when h.sched is set.
struct StepScalars {
    float lr, lrwd, bc1, bc2;
};

__device__ __forceinline__ StepScalars step_scalars(const AdamwScalars& h) {
    if (h.sched == nullptr) return StepScalars{h.lr, h.lrwd, h.bc1, h.bc2};
    const float lr = __ldg(h.sched);
    return StepScalars{lr, __fmul_rn(lr, h.wd), __ldg(h.sched + 1), __ldg(h.sched + 2)};
}

// The clipping coefficient, or 1 when no norm is given.
__device__ __forceinline__ float clip_coef(const AdamwScalars& h) {
    if (h.norm_sq == nullptr) return 1.0f;
    const double nrm = __dsqrt_rn(*h.norm_sq);
    const float c = __double2float_rn(__ddiv_rn((double)h.max_norm, __dadd_rn(nrm, 1e-6)));
    return c < 1.0f ? c : 1.0f;
}

// g is the mean gradient (already divided and clipped); st the step's scalars.
__device__ __forceinline__ void adamw_update(float g, float& w, float& m, float& v,
                                             const AdamwScalars& h, const StepScalars& st) {
    const float mi = __fadd_rn(__fmul_rn(h.b1, m), __fmul_rn(h.omb1, g));
    const float vi = __fadd_rn(__fmul_rn(h.b2, v), __fmul_rn(h.omb2, __fmul_rn(g, g)));
    const float m_hat = __fdiv_rn(mi, st.bc1);
    const float v_hat = __fdiv_rn(vi, st.bc2);
    float wi = __fsub_rn(w, __fmul_rn(st.lrwd, w));                       // decoupled decay
    const float denom = __fadd_rn(__fsqrt_rn(v_hat), h.eps);
    wi = __fsub_rn(wi, __fmul_rn(st.lr, __fdiv_rn(m_hat, denom)));         // Adam step
    w = wi;
    m = mi;
    v = vi;
}

// The mean gradient of one element from its source sum: the IEEE quotient
// sum / divisor, then the clip multiply (exact when coef == 1).  When the
// divisor is a power of two, sum * (1 / divisor) is the same correctly rounded
// value (both round the same real number once) at the cost of one multiply;
// kPow2 kernels take that branch (measured on GB300: +0.5-1 % for bf16
// sources, +2 % for 8-bit ones, but -5 % for the fp32-source update, which
// keeps the plain division).
template <bool kPow2 = false>
__device__ __forceinline__ float mean_grad(float sum, const AdamwScalars& h, float coef) {
    float g;
    if (ZGB_POW2_DIV && kPow2 && h.inv_divisor != 0.0f)
        g = __fmul_rn(sum, h.inv_divisor);
    else
        g = __fdiv_rn(sum, h.divisor);
    return __fmul_rn(g, coef);
}

// Update 8 elements at e from their source sums and loaded state; store the
// state and return the 8 bf16 results packed in a 16-byte vector.  P is a
// parameter block with the update target w, m, v and scalars h; sc is the
// step's scalars, resolved once per thread (step_scalars).
template <bool kPow2, class P>
__device__ __forceinline__ uint4 update_vec(const P& p, int64_t e, const float (&s)[8],
                                            const float4 (&st)[6], float coef, const StepScalars& sc) {
    float w[8] = {st[0].x, st[0].y, st[0].z, st[0].w, st[1].x, st[1].y, st[1].z, st[1].w};
    float m[8] = {st[2].x, st[2].y, st[2].z, st[2].w, st[3].x, st[3].y, st[3].z, st[3].w};
    float v[8] = {st[4].x, st[4].y, st[4].z, st[4].w, st[5].x, st[5].y, st[5].z, st[5].w};
#pragma unroll
    for (int j = 0; j < 8; ++j) adamw_update(mean_grad<kPow2>(s[j], p.h, coef), w[j], m[j], v[j], p.h, sc);
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
    return o;
}

// The same, storing the bf16 results at out + e.
template <bool kPow2, class P>
__device__ __forceinline__ void finish_vec(const P& p, int64_t e, const float (&s)[8],
                                           const float4 (&st)[6], float coef, const StepScalars& sc) {
    st_stream_u4(p.out + e, update_vec<kPow2>(p, e, s, st, coef, sc));
}

// The same with the 8-bit output: the bf16 results in the 8-bit block format
// (block 256) at qout + e, the block's scale at qscale[e / 256].  The 32 lanes
// of the calling warp must hold the 256 consecutive elements of one block
// (consecutive 8-element vectors, the first on a block boundary); codes and
// scale are computed exactly as by the quantizer (zero_quantize_int8).
template <bool kPow2, class P>
__device__ __forceinline__ void finish_vec_q8(const P& p, int64_t e, const float (&s)[8],
                                              const float4 (&st)[6], float coef, const StepScalars& sc,
                                              int8_t* qout, float* qscale) {
    const uint4 o = update_vec<kPow2>(p, e, s, st, coef, sc);
    const float a = warp_block_absmax(absmax8_bits(o, 0u));
    const float inv = a == 0.0f ? 0.0f : __fdiv_rn(127.0f, a);          // a zero block: codes 0
    *reinterpret_cast<uint2*>(qout + e) = quant8(o, inv);
    if ((threadIdx.x & 31) == 0) qscale[e >> 8] = __fdiv_rn(a, 127.0f);
}

template <class P>
__device__ __forceinline__ void load_state(const P& p, int64_t e, float4 (&st)[6]) {
    st[0] = ld_stream_f4(p.w + e);
    st[1] = ld_stream_f4(p.w + e + 4);
    st[2] = ld_stream_f4(p.m + e);
    st[3] = ld_stream_f4(p.m + e + 4);
    st[4] = ld_stream_f4(p.v + e);
    st[5] = ld_stream_f4(p.v + e + 4);
}

// The launch parameters of the fused update kernels.
struct UpdateParams {
    const void* src[ZERO_MAX_SRC];  // gradient sources (bf16 or fp32), offset to the range start
    const float* acc[ZERO_MAX_SRC]; // fp32 accumulators of the fused kinds, offset likewise
    float* w;
    float* m;
    float* v;
    uint16_t* out;                  // bf16 output, or nullptr when q is set
    int8_t* q;                      // 8-bit output (block 256) instead of bf16, or nullptr
    float* qscale;                  // its block scales, one per 256 elements
    int64_t n;                      // elements in the range
    int32_t n_src;                  // gradient sources (ranks)
    AdamwScalars h;
};

// ----------------------------------------------------------------- host

// The TMA-staged variant for bf16 sources (zero_rs_adamw_tma.cu): a status
// code, or 1 when it does not apply (a source count other than 1, 2, 4 or 8),
// so that the caller falls back to the register-staged kernel.  The caller
// only dispatches aligned ranges to it.
int launch_rs_adamw_tma(const UpdateParams& p, cudaStream_t stream);
// Reads and clears the device status word of the bounded waits (ZERO_OK or
// ZERO_ETIMEOUT); synchronizes the device.
int take_device_status();

// Where an update over flat [begin, end) of the owners rank_begin..rank_end-1
// reads and writes: state and output pointers already offset to `begin`.
struct UpdateTarget {
    float* w;
    float* m;
    float* v;
    uint16_t* out;  // nullptr for ZERO_OUT_NONE
    int64_t n;
    bool aligned;   // all pointers 16-byte aligned
};

// out_mode of an update whose output is not bf16 (internal: the 8-bit output).
constexpr int32_t ZERO_OUT_NONE = -1;

// Argument checks that need no CUDA call, then the offsets (zero_gb300.h,
// zero_reduce_scatter_adamw: state of i at [i - rank_begin*S]; out at [i] for
// ZERO_OUT_FULL, like the state for ZERO_OUT_SHARD).  A bf16 output
// (q8_out false) needs out_mode ZERO_OUT_FULL or ZERO_OUT_SHARD and a non-null
// out; only the library's 8-bit-output updates (q8_out true) pass
// ZERO_OUT_NONE with a null out, so no public argument reaches a null store.
int prepare_target(const zero_layout_t* L, int32_t rank_begin, int32_t rank_end, int64_t begin,
                   int64_t end, float* master, float* m, float* v, uint16_t* out, int32_t out_mode,
                   bool q8_out, UpdateTarget* t);
// The pointer-kind checks (CUDA calls) of a prepared target.
int check_target_ptrs(const UpdateTarget& t);
// Hyper-parameter checks and the fp32 scalars of the update.
int make_scalars(const zero_adamw_t* hp, float divisor, AdamwScalars* h);
// 1 - b1^t and 1 - b2^t in fp64 from the fp32 betas, rounded once to fp32.
void bias_corrections(float b1, float b2, int64_t t, float* bc1, float* bc2);
// Reads and clears the status word of zero_schedule_advance (ZERO_OK or
// ZERO_ERANGE); synchronizes the device.
int take_schedule_status();

}  // namespace zgb
