// The 8-bit gradient reduce-scatter (ZeRO++ quantized gradients), sm_103a.
//
// "ZeRO Optimizer, in depth", "Offload and ZeRO++" (zero_quantized_gradients
// quantises the gradient reduce-scatter) and "ZeRO and FSDP", "Fewer bytes on
// the wire".  Every rank has quantized its bf16 gradient slice for owner o in
// the block format of the weight gather (zero_quantize_int8 over the rank's
// whole gradient: slice o's codes at [o*S], its scales at [o*nb]).  For each
// owned element the owner reads the n_src codes (1 byte each) and their block
// scales, forms g_r = code * scale (one fp32 rounding), sums over ranks in
// ascending order from +0, and then
//   zero_reduce_scatter_adamw_int8     divides once, AdamW, bf16 cast, gather
//                                      write (what zero_reduce_scatter_adamw
//                                      does with the sum of bf16 gradients);
//   zero_reduce_scatter_adamw_int8_q8  the same with the owners' shards written
//                                      in the 8-bit block format instead of
//                                      bf16 (both ZeRO++ paths in one pass);
//   zero_accumulate_int8               adds the sum into an fp32 buffer (the
//                                      stage-3 layer reduce-scatter, or stage-2
//                                      accumulation).
// Bytes per element: n_src * (1 + 4/block) + 26 for the update, + 4 (+ 4 when
// adding) for the accumulation -- against 2 * n_src bytes of bf16 gradients.
//
// Design: the register-staged stream of the bf16 update.  A thread takes 8
// consecutive elements per vector: one 64-bit code load per source (a warp
// reads 256 consecutive bytes of each source), the source's block scale
// through the read-only path (blocks are >= 256 elements, so the 32 lanes of a
// warp share one scale), the fp32 state as 128-bit loads; every load of a
// vector is issued before the first add.  The scale index of an element is
// its owner's scale offset plus (slice-local index) >> log2(block).  A call
// over several whole shards is one launch with blockIdx.y = owner (every CTA
// inside one owner's slice); a call over several owners whose range cuts a
// shard is one launch over the whole range (kFlat), each vector finding its
// owner by comparing its index with a cached owner boundary; a call inside one
// owner's slice, or whose owner boundaries fall off the 8-element vector grid,
// is one launch per owner it meets.  The update with 8-bit output moves its
// fp32 state with 256-bit loads and stores where every slice's state starts on
// a 32-byte boundary (the other kinds measured slower with them); the update
// with bf16 output asks L2 for 256-byte blocks of the code streams.  Every
// kind loads the codes through the read-only path.
#include <cmath>

#include "zero_tma.cuh"
#include "zero_update.cuh"

#ifndef ZGB_QGRAD_WAVES
#define ZGB_QGRAD_WAVES 1    // update: grid = resident CTAs x this (measured: x1 +5 % over x64)
#endif
#ifndef ZGB_QACC_WAVES
#define ZGB_QACC_WAVES 1     // accumulation: the same (measured: 5.7 TB/s at x1, 5.2 at x64)
#endif
#ifndef ZGB_QGRAD_MULTI
#define ZGB_QGRAD_MULTI 1    // 1: a call over several whole shards is one launch (blockIdx.y =
                             // owner) when every slice takes the vector kernel; 0: one per owner
#endif
#ifndef ZGB_QGRAD_MINBLOCKS
#define ZGB_QGRAD_MINBLOCKS 3 // update with one vector per thread: CTAs per SM the register
                              // allocation must allow (3: 80 registers, no spills); the others keep
                              // 2 (they spill below 128)
#endif
#ifndef ZGB_QACC_MINBLOCKS
#define ZGB_QACC_MINBLOCKS 0  // the same for the accumulation; 0 = 3 with one vector per thread
                              // (measured +1.5 % at 8 sources), else 2
#endif
#ifndef ZGB_QGRAD_U
#define ZGB_QGRAD_U 0        // vectors per thread and iteration; 0 = the measured choice
#endif
#ifndef ZGB_QACC_U
#define ZGB_QACC_U 0         // the same for the accumulation
#endif
#ifndef ZGB_QFLAT_WAVES
#define ZGB_QFLAT_WAVES 8    // kFlat launches: grid = resident CTAs x this (measured on GPT-2-XL
                             // buckets: 6546 GB/s at x8 against 6471 at x1)
#endif
#ifndef ZGB_QGRAD_FLAT
#define ZGB_QGRAD_FLAT 1     // a call over several owners' slices as one launch over its whole
                             // range, each vector finding its owner (kFlat): 0 never, 1 for
                             // ranges that cut shards only, 2 for every multi-owner call
#endif
#ifndef ZGB_QV8
#define ZGB_QV8 4            // 256-bit accesses to the fp32 state (update) or destination
                             // (accumulation) where every slice's start is 32-byte aligned: bit 0
                             // the accumulation, bit 1 the update, bit 2 the update with 8-bit
                             // output (measured on the Llama-7B units: 8-bit output +2.4 %,
                             // 6588 against 6434 GB/s; the update -2.3 %, the accumulation -0.4 %)
#endif
#ifndef ZGB_QCODE_PF256
#define ZGB_QCODE_PF256 2    // code loads that ask L2 for the enclosing 256 bytes: bit 0 the
                             // accumulation, bit 1 the update, bit 2 the update with 8-bit output
                             // (measured: the update +0.8 %, 6589 against 6537 GB/s on GPT-2-XL
                             // buckets; the others within 0.2 %, and 128 bytes changed nothing)
#endif
#ifndef ZGB_QACC_ST_PLAIN
#define ZGB_QACC_ST_PLAIN 1  // the accumulation's fp32 result stored with the default cache policy
                             // instead of evict-first, so that the part still in L2 serves the
                             // update that reads it next (measured on the Llama-7B units: +0.9 %,
                             // 6347 against 6292 GB/s, the update after it +0.1 %)
#endif
#ifndef ZGB_QWS
#define ZGB_QWS 0            // opt-in: the code streams staged by bulk copies (qgrad_ws_kernel)
                             // for 1, 2, 4 or 8 sources with 16-byte aligned slices: bit 0 the
                             // accumulation, bit 1 the updates.  Bit-exact, but measured slower
                             // than the register-staged kernels (update 6093 against 6350 GB/s,
                             // accumulation 6133 against 6292, 8-bit output 6115 against 6432)
#endif
#ifndef ZGB_QWS_STAGES
#define ZGB_QWS_STAGES 4     // stages of its ring per CTA
#endif
#ifndef ZGB_QWS_MINBLOCKS
#define ZGB_QWS_MINBLOCKS 2  // CTAs per SM its register allocation must allow
#endif
#ifndef ZGB_QWS_TIMEOUT_CYCLES
#define ZGB_QWS_TIMEOUT_CYCLES (1ll << 31)   // SM cycles before a wait gives up (~1 s)
#endif

namespace zgb {

// One launch covers one owner's slice (owners == 0: n, k0 describe it, every
// pointer is offset to its first element) or, with owners > 0, the slices of
// owners o_first .. o_first + owners - 1 that meet [begin, end), one per
// blockIdx.y (every pointer offset to `begin`, the scale pointers to the
// start of the sources' scale arrays), or, with owners < 0 (the kFlat
// kernels), the whole range [begin, end) as one stream of vectors, pointers
// as for owners > 0, each vector's owner found from its flat index.
struct QGradParams {
    const int8_t* q[ZERO_MAX_SRC];     // rank r's codes
    const float* scale[ZERO_MAX_SRC];  // rank r's block scales (of this owner's slice if owners == 0)
    float* w;                          // update: state, offset like q
    float* m;
    float* v;
    uint16_t* out;                     // update: bf16 output, offset like q
    float* dst;                        // accumulation: fp32 destination, offset like q
    int8_t* qout;                      // update with 8-bit output: codes, offset like w
    float* qoscale;                    // and their block scales (one per 256 elements)
    int64_t n;                         // owners == 0: elements of the launch, in one owner's slice
    int64_t k0;                        // owners == 0: slice-local index of its first element
    int64_t begin, end;                // owners > 0: the flat range of the call
    int64_t S;                         // owners > 0: shard length
    int64_t nb;                        // owners > 0: scale blocks per shard
    int32_t o_first;                   // owners > 0: the first owner
    int32_t owners;
    int32_t n_src;
    int32_t block_shift;               // log2(block)
    int32_t first;                     // accumulation: 1 overwrites dst, 0 adds to it
    int32_t v8;                        // every slice's state (or dst) start is 32-byte aligned
    AdamwScalars h;
};

// The slice a CTA works on.  eoff: its first element's offset from the code
// and target pointers; k0: that element's slice-local index (the block grid);
// n: its length; soff: the offset of its scales from the scale pointers.
struct QSlice {
    int64_t eoff, k0, n, soff;
};

__device__ __forceinline__ QSlice qslice(const QGradParams& p) {
    if (p.owners == 0) return QSlice{0, p.k0, p.n, 0};
    if (p.owners < 0) return QSlice{0, 0, p.n, 0};     // kFlat: the whole range, owners per vector
    const int64_t o = (int64_t)p.o_first + blockIdx.y;
    const int64_t lo = p.begin > o * p.S ? p.begin : o * p.S;
    const int64_t hi = p.end < (o + 1) * p.S ? p.end : (o + 1) * p.S;
    return QSlice{lo - p.begin, lo - o * p.S, hi - lo, o * p.nb};
}

// kFlat: the owner slice that holds the last vector a thread looked up:
// flat element i lies in [lo, hi) = [o*S, (o+1)*S), and owner o's scales start
// at soff = o*nb.  A thread's vectors advance by the grid's stride, far less
// than a shard, so the 64-bit division that finds an owner runs about once
// per owner a thread meets.
struct OwnerCache {
    int64_t lo = 0, hi = 0, soff = 0;
};

// The slice of vector (or element) e: the launch's own, or with kFlat the
// owner's that holds flat element begin + sl.eoff + e, as a QSlice with the
// same eoff whose k0 + e is that element's slice-local index.
template <bool kFlat>
__device__ __forceinline__ QSlice slice_of(const QGradParams& p, const QSlice& sl, int64_t e, OwnerCache& c) {
    if constexpr (!kFlat) return sl;
    const int64_t i = p.begin + sl.eoff + e;
    if (i < c.lo || i >= c.hi) {
        const int64_t o = i / p.S;
        c.lo = o * p.S;
        c.hi = c.lo + p.S;
        c.soff = o * p.nb;
    }
    return QSlice{sl.eoff, p.begin + sl.eoff - c.lo, sl.n, c.soff};
}

// Code j (0..3) of a 32-bit word as an fp32 value (exact: |code| <= 127).
__device__ __forceinline__ float code_f32(uint32_t word, int j) {
    return (float)(int)(int8_t)(word >> (8 * j));
}

// Whether a kernel kind takes the 256-bit accesses (ZGB_QV8).
template <bool kUpdate, bool kQ8>
__host__ __device__ constexpr bool qgrad_v8() {
    return (ZGB_QV8 & (kQ8 ? 4 : kUpdate ? 2 : 1)) != 0;
}

#if ZGB_QV8
// 256-bit evict-first accesses (sm_100 and later); p 32-byte aligned.
__device__ __forceinline__ void ld_v8(const float* p, float4& a, float4& b) {
    asm volatile("ld.global.cs.v8.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=f"(a.x), "=f"(a.y), "=f"(a.z), "=f"(a.w), "=f"(b.x), "=f"(b.y), "=f"(b.z), "=f"(b.w)
                 : "l"(p));
}
__device__ __forceinline__ void st_v8(float* p, const float (&x)[8]) {
    asm volatile("st.global.cs.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                 :: "l"(p), "f"(x[0]), "f"(x[1]), "f"(x[2]), "f"(x[3]), "f"(x[4]), "f"(x[5]), "f"(x[6]), "f"(x[7])
                 : "memory");
}
#endif

// One lane's 8 codes of a source: evict-first, or through the read-only path
// for the kinds in ZGB_QCODE_NC; for the kinds in ZGB_QCODE_PF256 the miss
// fetches the enclosing 256-byte block into L2 (the warp reads 256
// consecutive bytes of each source).
#ifndef ZGB_QCODE_NC
#define ZGB_QCODE_NC 7       // code loads through the read-only path (ld.global.nc; no kernel
                             // writes codes) instead of evict-first: bit 0 the accumulation, bit 1
                             // the update, bit 2 the update with 8-bit output (measured: the
                             // accumulation +1.2 %, 6421 against 6347 GB/s on the Llama-7B units;
                             // the update +1.7 %, 6714 against 6603 on GPT-2-XL buckets; the 8-bit
                             // output +2.0 %, 6723 against 6588)
#endif
template <bool kUpdate, bool kQ8>
__device__ __forceinline__ uint2 ld_codes(const int8_t* p) {
    constexpr int kBit = kQ8 ? 4 : kUpdate ? 2 : 1;
    uint2 c;
    if constexpr ((ZGB_QCODE_NC & kBit) != 0 && (ZGB_QCODE_PF256 & kBit) != 0) {
        asm volatile("ld.global.nc.L2::256B.v2.u32 {%0, %1}, [%2];" : "=r"(c.x), "=r"(c.y) : "l"(p));
    } else if constexpr ((ZGB_QCODE_NC & kBit) != 0) {
        c = __ldg(reinterpret_cast<const uint2*>(p));
    } else if constexpr ((ZGB_QCODE_PF256 & kBit) != 0) {
        asm volatile("ld.global.cs.L2::256B.v2.u32 {%0, %1}, [%2];" : "=r"(c.x), "=r"(c.y) : "l"(p));
    } else {
        c = ld_stream_u2(p);
    }
    return c;
}

// x[j] = x[j] + code_j * scale for the 8 codes of c; each product and each
// sum one IEEE rounding.
__device__ __forceinline__ void add_codes8(float (&x)[8], const uint2 c, const float s) {
#pragma unroll
    for (int j = 0; j < 4; ++j) x[j] = __fadd_rn(x[j], __fmul_rn(code_f32(c.x, j), s));
#pragma unroll
    for (int j = 0; j < 4; ++j) x[4 + j] = __fadd_rn(x[4 + j], __fmul_rn(code_f32(c.y, j), s));
}

// One vector's loads: R sources' codes and scales, then the state (update) or
// the destination (accumulation that adds).
template <int R, bool kUpdate>
struct QVec {
    uint2 c[R];
    float s[R];
    float4 st[kUpdate ? 6 : 2];
};

// e: the element's index in the slice.
template <int R, bool kUpdate, bool kQ8>
__device__ __forceinline__ void load_qvec(const QGradParams& p, const QSlice& sl, int64_t e,
                                          QVec<R, kUpdate>& x) {
    const int64_t b = sl.soff + ((sl.k0 + e) >> p.block_shift);
    const int64_t g = sl.eoff + e;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        x.c[r] = ld_codes<kUpdate, kQ8>(p.q[r] + g);
        x.s[r] = __ldg(p.scale[r] + b);
    }
#if ZGB_QV8
    if (qgrad_v8<kUpdate, kQ8>() && p.v8) {
        if constexpr (kUpdate) {
            ld_v8(p.w + g, x.st[0], x.st[1]);
            ld_v8(p.m + g, x.st[2], x.st[3]);
            ld_v8(p.v + g, x.st[4], x.st[5]);
        } else if (!p.first) {
            ld_v8(p.dst + g, x.st[0], x.st[1]);
        }
        return;
    }
#endif
    if constexpr (kUpdate) {
        load_state(p, g, x.st);
    } else if (!p.first) {
        x.st[0] = ld_stream_f4(p.dst + g);
        x.st[1] = ld_stream_f4(p.dst + g + 4);
    }
}

// The accumulation's result of one vector: (dst +) the source sum; e indexes
// from the target pointers.
__device__ __forceinline__ void store_acc(const QGradParams& p, int64_t e, float (&x)[8],
                                          const float4 (&d)[2]) {
    if (!p.first) {
        const float4 a = d[0], b = d[1];
        x[0] = __fadd_rn(a.x, x[0]); x[1] = __fadd_rn(a.y, x[1]);
        x[2] = __fadd_rn(a.z, x[2]); x[3] = __fadd_rn(a.w, x[3]);
        x[4] = __fadd_rn(b.x, x[4]); x[5] = __fadd_rn(b.y, x[5]);
        x[6] = __fadd_rn(b.z, x[6]); x[7] = __fadd_rn(b.w, x[7]);
    }
#if ZGB_QACC_ST_PLAIN
    *reinterpret_cast<float4*>(p.dst + e) = make_float4(x[0], x[1], x[2], x[3]);
    *reinterpret_cast<float4*>(p.dst + e + 4) = make_float4(x[4], x[5], x[6], x[7]);
#else
    st_stream_f4(p.dst + e, make_float4(x[0], x[1], x[2], x[3]));
    st_stream_f4(p.dst + e + 4, make_float4(x[4], x[5], x[6], x[7]));
#endif
}

#if ZGB_QV8
// update_vec of the fused update with 256-bit state stores (the same
// element arithmetic, so the same results).
__device__ __forceinline__ uint4 update_vec_v8(const QGradParams& p, int64_t e, const float (&s)[8],
                                               const float4 (&st)[6], const StepScalars& sc) {
    float w[8] = {st[0].x, st[0].y, st[0].z, st[0].w, st[1].x, st[1].y, st[1].z, st[1].w};
    float m[8] = {st[2].x, st[2].y, st[2].z, st[2].w, st[3].x, st[3].y, st[3].z, st[3].w};
    float v[8] = {st[4].x, st[4].y, st[4].z, st[4].w, st[5].x, st[5].y, st[5].z, st[5].w};
#pragma unroll
    for (int j = 0; j < 8; ++j) adamw_update(mean_grad<true>(s[j], p.h, 1.0f), w[j], m[j], v[j], p.h, sc);
    st_v8(p.w + e, w);
    st_v8(p.m + e, m);
    st_v8(p.v + e, v);
    uint4 o;
    o.x = pack_bf16x2(w[0], w[1]);
    o.y = pack_bf16x2(w[2], w[3]);
    o.z = pack_bf16x2(w[4], w[5]);
    o.w = pack_bf16x2(w[6], w[7]);
    return o;
}
#endif

// One vector's result from its loads x: the source sum, then the update
// (bf16 or 8-bit output) or the accumulation; e indexes from the target
// pointers.
template <int R, bool kUpdate, bool kQ8>
__device__ __forceinline__ void qgrad_finish(const QGradParams& p, int64_t e, QVec<R, kUpdate>& x,
                                             const StepScalars& sc) {
    float s[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) s[j] = 0.0f;
#pragma unroll
    for (int r = 0; r < R; ++r) add_codes8(s, x.c[r], x.s[r]);
#if ZGB_QV8
    if (qgrad_v8<kUpdate, kQ8>() && p.v8) {
        if constexpr (kQ8) {            // finish_vec_q8 with the state stored by update_vec_v8
            const uint4 o = update_vec_v8(p, e, s, x.st, sc);
            const float a = warp_block_absmax(absmax8_bits(o, 0u));
            const float inv = a == 0.0f ? 0.0f : __fdiv_rn(127.0f, a);
            *reinterpret_cast<uint2*>(p.qout + e) = quant8(o, inv);
            if ((threadIdx.x & 31) == 0) p.qoscale[e >> 8] = __fdiv_rn(a, 127.0f);
        } else if constexpr (kUpdate) {
            st_stream_u4(p.out + e, update_vec_v8(p, e, s, x.st, sc));
        } else {
            if (!p.first) {
                s[0] = __fadd_rn(x.st[0].x, s[0]); s[1] = __fadd_rn(x.st[0].y, s[1]);
                s[2] = __fadd_rn(x.st[0].z, s[2]); s[3] = __fadd_rn(x.st[0].w, s[3]);
                s[4] = __fadd_rn(x.st[1].x, s[4]); s[5] = __fadd_rn(x.st[1].y, s[5]);
                s[6] = __fadd_rn(x.st[1].z, s[6]); s[7] = __fadd_rn(x.st[1].w, s[7]);
            }
            st_v8(p.dst + e, s);
        }
        return;
    }
#endif
    if constexpr (kQ8) {
        finish_vec_q8<true>(p, e, s, x.st, 1.0f, sc, p.qout, p.qoscale);
    } else if constexpr (kUpdate) {
        finish_vec<true>(p, e, s, x.st, 1.0f, sc);
    } else {
        const float4 d[2] = {x.st[0], x.st[1]};
        store_acc(p, e, s, d);
    }
}

// U vectors (vi0, vi0 + kThreads, ...) with a compile-time source count.
template <int R, bool kUpdate, int U, bool kQ8, bool kFlat>
__device__ __forceinline__ void qgrad_vecs(const QGradParams& p, const QSlice& sl, int64_t vi0,
                                           int64_t nv, const StepScalars& sc, OwnerCache& oc) {
    QVec<R, kUpdate> x[U];
    bool ok[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int64_t vi = vi0 + u * kThreads;
        ok[u] = vi < nv;
        if (ok[u]) load_qvec<R, kUpdate, kQ8>(p, slice_of<kFlat>(p, sl, vi * 8, oc), vi * 8, x[u]);
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
        if (ok[u]) qgrad_finish<R, kUpdate, kQ8>(p, sl.eoff + (vi0 + u * kThreads) * 8, x[u], sc);
}

// One vector with a runtime source count, one source at a time.
template <bool kUpdate, bool kQ8>
__device__ __forceinline__ void qgrad_vec_dyn(const QGradParams& p, const QSlice& sl, int64_t vi,
                                              const StepScalars& sc) {
    const int64_t b = sl.soff + ((sl.k0 + vi * 8) >> p.block_shift);   // sl: the vector's slice
    const int64_t e = sl.eoff + vi * 8;
    float s[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) s[j] = 0.0f;
    for (int r = 0; r < p.n_src; ++r) add_codes8(s, ld_stream_u2(p.q[r] + e), __ldg(p.scale[r] + b));
    if constexpr (kUpdate) {
        float4 st[6];
        load_state(p, e, st);
        if constexpr (kQ8)
            finish_vec_q8<true>(p, e, s, st, 1.0f, sc, p.qout, p.qoscale);
        else
            finish_vec<true>(p, e, s, st, 1.0f, sc);
    } else {
        float4 d[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
        if (!p.first) {
            d[0] = ld_stream_f4(p.dst + e);
            d[1] = ld_stream_f4(p.dst + e + 4);
        }
        store_acc(p, e, s, d);
    }
}

// One element (ragged tails, ranges off the 8-element grid).
// i: the element's index in the slice.
template <bool kUpdate>
__device__ __forceinline__ void qgrad_one(const QGradParams& p, const QSlice& sl, int64_t il,
                                          const StepScalars& sc) {
    const int64_t b = sl.soff + ((sl.k0 + il) >> p.block_shift);
    const int64_t i = sl.eoff + il;
    float s = 0.0f;
    for (int r = 0; r < p.n_src; ++r) s = __fadd_rn(s, __fmul_rn((float)p.q[r][i], __ldg(p.scale[r] + b)));
    if constexpr (kUpdate) {
        float w = p.w[i], m = p.m[i], v = p.v[i];
        adamw_update(mean_grad(s, p.h, 1.0f), w, m, v, p.h, sc);
        p.w[i] = w;
        p.m[i] = m;
        p.v[i] = v;
        p.out[i] = to_bf16(w);
    } else {
        p.dst[i] = p.first ? s : __fadd_rn(p.dst[i], s);
    }
}

// Vectors per thread and iteration: the code loads are 8 bytes, so a vector
// with few sources leaves HBM short of bytes in flight unless a thread takes
// several.
template <int R, bool kUpdate>
__host__ __device__ constexpr int qgrad_vectors_per_iter() {
    return R == 0 ? 1
         : kUpdate ? (ZGB_QGRAD_U > 0 ? ZGB_QGRAD_U : R <= 2 ? 2 : 1)
                   : (ZGB_QACC_U > 0 ? ZGB_QACC_U : R <= 4 ? 4 : 1);
}

// CTAs per SM the register allocation must allow.
template <int R, bool kUpdate>
__host__ __device__ constexpr int qgrad_min_blocks() {
    return kUpdate ? (qgrad_vectors_per_iter<R, kUpdate>() == 1 ? ZGB_QGRAD_MINBLOCKS : 2)
                   : (ZGB_QACC_MINBLOCKS > 0 ? ZGB_QACC_MINBLOCKS
                      : qgrad_vectors_per_iter<R, kUpdate>() == 1 ? 3 : 2);
}

// kQ8 (with kUpdate): the output is 8-bit codes and block scales (p.qout,
// p.qoscale) instead of bf16; the host guarantees whole 256-element blocks.
// kFlat: the launch covers [begin, end) as one stream (p.owners < 0), each
// vector's owner looked up; the host takes it only when every owner boundary
// lies on the launch's 8-element vector grid.
template <int R, bool kUpdate, bool kQ8 = false, bool kFlat = false>
__global__ void __launch_bounds__(kThreads, (qgrad_min_blocks<R, kUpdate>()))
qgrad_vec_kernel(const __grid_constant__ QGradParams p) {
    const StepScalars sc = kUpdate ? step_scalars(p.h) : StepScalars{};
    const QSlice sl = qslice(p);
    const int64_t nv = sl.n >> 3;
    const int64_t tid = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    OwnerCache oc;
    if constexpr (R > 0) {
        constexpr int U = qgrad_vectors_per_iter<R, kUpdate>();
        const int64_t chunk = (int64_t)U * kThreads;
        for (int64_t v0 = (int64_t)blockIdx.x * chunk + threadIdx.x; v0 < nv; v0 += (int64_t)gridDim.x * chunk)
            qgrad_vecs<R, kUpdate, U, kQ8, kFlat>(p, sl, v0, nv, sc, oc);
    } else {
        const int64_t stride = (int64_t)gridDim.x * kThreads;
        for (int64_t vi = tid; vi < nv; vi += stride)
            qgrad_vec_dyn<kUpdate, kQ8>(p, slice_of<kFlat>(p, sl, vi * 8, oc), vi, sc);
    }
    if constexpr (!kQ8) {
        const int64_t tail = sl.n - (nv << 3);
        if (tid < tail) qgrad_one<kUpdate>(p, slice_of<kFlat>(p, sl, (nv << 3) + tid, oc), (nv << 3) + tid, sc);
    }
}

template <bool kUpdate>
__global__ void __launch_bounds__(kThreads) qgrad_scalar_kernel(const __grid_constant__ QGradParams p) {
    const StepScalars sc = kUpdate ? step_scalars(p.h) : StepScalars{};
    const QSlice sl = qslice(p);
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < sl.n; i += stride)
        qgrad_one<kUpdate>(p, sl, i, sc);
}

// ----------------------------------------------------------------------------
// Warp-specialized variant: the code streams staged by bulk copies.
//
// The register-staged kernel above holds 8 bytes of codes per source in flight
// per thread and waits for them before it computes, so the SM's bytes in
// flight fall with every pass's compute.  Here warp 0's lane 0 (the producer)
// copies tile k's R code streams -- kQWsTile bytes each, 1-D bulk copies
// (cp.async.bulk) -- into stage k % S of a shared-memory ring, arming the
// stage's "full" mbarrier with the byte count, once every consumer warp has
// released the stage's previous tile (its "empty" mbarrier, one arrival per
// consumer warp).  Consumer warps 1..C each own 256 consecutive elements of a
// tile, 8 per lane: they load their block scales and (for the update) their
// fp32 state or (for an accumulation that adds) their fp32 destination
// before waiting on the stage, read their codes from it, release it, and then
// compute and store exactly as the register-staged kernel does -- the same
// functions, so the results are bit-identical.  No CTA-wide barrier sits in
// the loop.  Tile u of a stage completes phase u of both barriers; waits pass
// the parity u & 1 (the producer cannot refill a stage before every consumer
// released it, and a consumer cannot release a tile that was not issued, so no
// wait trails by two phases).
//
// Bulk copies start on 16-byte boundaries and move multiples of 16 bytes: the
// host takes this kernel only when every source's slice starts 16-byte
// aligned; the tiles cover the first n16 = n & ~15 elements of the slice, and
// the last n - n16 (< 16) go element by element to CTA 0's first consumer warp.
//
// Every wait is bounded: a wait that gives up records ZERO_ETIMEOUT in
// g_qgrad_status (read by zero_status_check) and ends that warp's loop; the
// producer then waits, bounded again, for the copies of the last S tiles it
// issued, so that no copy lands in the shared memory of a finished CTA.
// ----------------------------------------------------------------------------

__device__ int g_qgrad_status;   // ZERO_OK, or ZERO_ETIMEOUT once a bounded wait gave up

constexpr int kQWsConsumers = 8;
constexpr int kQWsThreads = 32 * (kQWsConsumers + 1);
constexpr int kQWsTile = 256 * kQWsConsumers;        // elements (= bytes per source) per tile
constexpr int kQWsStages = ZGB_QWS_STAGES;
static_assert(kQWsStages >= 2 && kQWsStages <= 8, "the code ring runs with 2 to 8 stages");
static_assert(kQWsTile % 256 == 0, "a consumer warp's 256 elements must be whole 8-bit blocks");

template <int R>
constexpr uint32_t qws_smem_bytes() {
    return (uint32_t)(R * kQWsTile * kQWsStages);
}
static_assert(qws_smem_bytes<8>() <= 227 * 1024, "the ring must fit the shared memory of one CTA");

template <int R, bool kUpdate, bool kQ8>
__global__ void __launch_bounds__(kQWsThreads, ZGB_QWS_MINBLOCKS)
qgrad_ws_kernel(const __grid_constant__ QGradParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) uint64_t full[kQWsStages];
    __shared__ __align__(8) uint64_t empty[kQWsStages];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const QSlice sl = qslice(p);
    const int64_t n16 = sl.n & ~(int64_t)15;
    const int64_t n_tiles = (n16 + kQWsTile - 1) / kQWsTile;
    const int64_t count = blockIdx.x < n_tiles ? (n_tiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    auto tile_e0 = [&](int64_t k) { return ((int64_t)blockIdx.x + k * gridDim.x) * kQWsTile; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kQWsStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kQWsConsumers);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (warp == 0) {
        if (lane == 0) {
            int64_t k = 0;
            for (; k < count; ++k) {
                const int s = (int)(k % kQWsStages);
                if (k >= kQWsStages &&
                    !mbar_wait_bounded(&empty[s], (uint32_t)((k / kQWsStages - 1) & 1), ZGB_QWS_TIMEOUT_CYCLES)) {
                    atomicExch(&g_qgrad_status, ZERO_ETIMEOUT);
                    break;
                }
                const int64_t e0 = tile_e0(k);
                const uint32_t bytes = (uint32_t)min((int64_t)kQWsTile, n16 - e0);   // a multiple of 16
                unsigned char* st = smem + (size_t)s * R * kQWsTile;
                mbar_arrive_expect_tx(&full[s], bytes * (uint32_t)R);
#pragma unroll
                for (int r = 0; r < R; ++r)
                    bulk_g2s(st + r * kQWsTile, p.q[r] + sl.eoff + e0, bytes, &full[s]);
            }
            // the copies of the last stages issued must land before the CTA ends
            for (int64_t j = k > kQWsStages ? k - kQWsStages : 0; j < k; ++j)
                (void)mbar_wait_bounded(&full[j % kQWsStages], (uint32_t)((j / kQWsStages) & 1),
                                        ZGB_QWS_TIMEOUT_CYCLES);
        }
        return;
    }
    const StepScalars sc = kUpdate ? step_scalars(p.h) : StepScalars{};
    const int off = (warp - 1) * 256 + lane * 8;          // this lane's first element in a tile
    for (int64_t k = 0; k < count; ++k) {
        const int s = (int)(k % kQWsStages);
        const int64_t e0 = tile_e0(k);
        const bool act = off < min((int64_t)kQWsTile, n16 - e0);
        const int64_t e = e0 + off;                         // slice-local index
        const int64_t g = sl.eoff + e;                      // index from the code and target pointers
        float scale[R];
        float4 st[kUpdate ? 6 : 2];
        if (act) {
            const int64_t b = sl.soff + ((sl.k0 + e) >> p.block_shift);
#pragma unroll
            for (int r = 0; r < R; ++r) scale[r] = __ldg(p.scale[r] + b);
            if constexpr (kUpdate) {
                load_state(p, g, st);
            } else if (!p.first) {
                st[0] = ld_stream_f4(p.dst + g);
                st[1] = ld_stream_f4(p.dst + g + 4);
            }
        }
        const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full[s], (uint32_t)((k / kQWsStages) & 1),
                                                                  ZGB_QWS_TIMEOUT_CYCLES));
        if (!ok) {
            if (lane == 0) atomicExch(&g_qgrad_status, ZERO_ETIMEOUT);
            break;
        }
        uint2 c[R];
        if (act) {
            const unsigned char* stage = smem + (size_t)s * R * kQWsTile + off;
#pragma unroll
            for (int r = 0; r < R; ++r) c[r] = *reinterpret_cast<const uint2*>(stage + r * kQWsTile);
        }
        __syncwarp();                                        // the warp is done with stage s
        if (lane == 0) mbar_arrive(&empty[s]);
        if (act) {
            float x[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) x[j] = 0.0f;
#pragma unroll
            for (int r = 0; r < R; ++r) add_codes8(x, c[r], scale[r]);
            if constexpr (kQ8) {
                finish_vec_q8<true>(p, g, x, st, 1.0f, sc, p.qout, p.qoscale);
            } else if constexpr (kUpdate) {
                finish_vec<true>(p, g, x, st, 1.0f, sc);
            } else {
                const float4 d[2] = {st[0], st[1]};
                store_acc(p, g, x, d);
            }
        }
    }
    // the last n - n16 elements of the slice, element by element
    if constexpr (!kQ8) {
        if (blockIdx.x == 0 && warp == 1 && lane < sl.n - n16) qgrad_one<kUpdate>(p, sl, n16 + lane, sc);
    }
}

// Reads and clears the status word of the bounded waits above (ZERO_OK or
// ZERO_ETIMEOUT); synchronizes the device.
int take_qgrad_status() {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_qgrad_status, sizeof v) != cudaSuccess) {
        (void)cudaGetLastError();
        return ZERO_ECUDA;
    }
    if (v != ZERO_OK) {
        const int zero = ZERO_OK;
        if (cudaMemcpyToSymbol(g_qgrad_status, &zero, sizeof zero) != cudaSuccess) {
            (void)cudaGetLastError();
            return ZERO_ECUDA;
        }
    }
    return v == ZERO_OK ? ZERO_OK : ZERO_ETIMEOUT;
}

template <int R, bool kUpdate, bool kQ8>
int launch_qgrad_ws(const QGradParams& p, int64_t slice_max, cudaStream_t s) {
    const uint32_t smem = qws_smem_bytes<R>();
    const void* fn = (const void*)qgrad_ws_kernel<R, kUpdate, kQ8>;
    const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        note_cuda_error(e);
        return ZERO_ECUDA;
    }
    const int occupancy = ctas_per_sm(fn, kQWsThreads, smem);
    const int64_t slices = p.owners > 0 ? p.owners : 1;
    const int64_t cap = (int64_t)sm_count() * (occupancy > 0 ? occupancy : 1) / slices;
    const int64_t tiles = ((slice_max & ~(int64_t)15) + kQWsTile - 1) / kQWsTile;
    const dim3 grid((unsigned)(tiles < 1 ? 1 : (tiles < cap ? tiles : (cap > 0 ? cap : 1))), (unsigned)slices);
    qgrad_ws_kernel<R, kUpdate, kQ8><<<grid, kQWsThreads, smem, s>>>(p);
    return launch_status();
}

// Whether a launch of this kind takes the warp-specialized kernel.
template <bool kUpdate>
bool qgrad_ws_enabled() {
    return (ZGB_QWS & (kUpdate ? 2 : 1)) != 0;
}

// p.owners == 0: one owner's slice of p.n elements; else `owners` slices of
// at most `slice_max` elements, one per blockIdx.y, sharing the grid's CTAs.
template <int R, bool kUpdate, bool kQ8 = false>
int launch_qgrad_vec(const QGradParams& p, int64_t slice_max, cudaStream_t s) {
    if (p.owners < 0) {                       // one stream over the whole range
        const int occ = ctas_per_sm((const void*)qgrad_vec_kernel<R, kUpdate, kQ8, true>, kThreads, 0);
        const int64_t per = (int64_t)(R > 0 ? qgrad_vectors_per_iter<R, kUpdate>() : 1) * kThreads;
        const unsigned grid = grid_for(p.n >> 3, per, (int64_t)sm_count() * occ * ZGB_QFLAT_WAVES);
        qgrad_vec_kernel<R, kUpdate, kQ8, true><<<grid, kThreads, 0, s>>>(p);
        return launch_status();
    }
    const int occupancy = ctas_per_sm((const void*)qgrad_vec_kernel<R, kUpdate, kQ8>, kThreads, 0);
    const int64_t per_cta = (int64_t)qgrad_vectors_per_iter<R, kUpdate>() * kThreads;
    const int64_t waves = kUpdate ? ZGB_QGRAD_WAVES : ZGB_QACC_WAVES;
    const int64_t slices = p.owners > 0 ? p.owners : 1;
    const int64_t cap = (int64_t)sm_count() * occupancy * waves / slices;
    const dim3 grid(grid_for(slice_max >> 3, per_cta, cap > 0 ? cap : 1), (unsigned)slices);
    qgrad_vec_kernel<R, kUpdate, kQ8><<<grid, kThreads, 0, s>>>(p);
    return launch_status();
}

// vec: every slice of the launch takes the vector kernel (8-aligned slice
// starts, aligned pointers); the scalar kernel serves single-owner launches.
template <bool kUpdate, bool kQ8 = false>
int launch_qgrad(const QGradParams& p, bool vec, bool ws, int64_t slice_max, cudaStream_t s) {
    if (vec && ws && p.owners >= 0 && qgrad_ws_enabled<kUpdate>()) {
        switch (p.n_src) {
            case 1: return launch_qgrad_ws<1, kUpdate, kQ8>(p, slice_max, s);
            case 2: return launch_qgrad_ws<2, kUpdate, kQ8>(p, slice_max, s);
            case 4: return launch_qgrad_ws<4, kUpdate, kQ8>(p, slice_max, s);
            case 8: return launch_qgrad_ws<8, kUpdate, kQ8>(p, slice_max, s);
            default: break;                 // the register-staged kernels below
        }
    }
    if constexpr (kQ8) {                 // vector kernels only: whole 256-element blocks per warp
        if (!vec) return ZERO_EALIGN;
        switch (p.n_src) {
            case 1: return launch_qgrad_vec<1, kUpdate, true>(p, slice_max, s);
            case 2: return launch_qgrad_vec<2, kUpdate, true>(p, slice_max, s);
            case 4: return launch_qgrad_vec<4, kUpdate, true>(p, slice_max, s);
            case 8: return launch_qgrad_vec<8, kUpdate, true>(p, slice_max, s);
            default: return launch_qgrad_vec<0, kUpdate, true>(p, slice_max, s);
        }
    }
    if (!vec) {
        if (p.owners != 0) return ZERO_EINVAL;   // not reached: multi-owner launches are vector only
        const int occupancy = ctas_per_sm((const void*)qgrad_scalar_kernel<kUpdate>, kThreads, 0);
        const unsigned grid = grid_for(p.n, kThreads, (int64_t)sm_count() * occupancy);
        qgrad_scalar_kernel<kUpdate><<<grid, kThreads, 0, s>>>(p);
        return launch_status();
    }
    switch (p.n_src) {
        case 1: return launch_qgrad_vec<1, kUpdate>(p, slice_max, s);
        case 2: return launch_qgrad_vec<2, kUpdate>(p, slice_max, s);
        case 4: return launch_qgrad_vec<4, kUpdate>(p, slice_max, s);
        case 8: return launch_qgrad_vec<8, kUpdate>(p, slice_max, s);
        case 16: return launch_qgrad_vec<16, kUpdate>(p, slice_max, s);
        default: return launch_qgrad_vec<0, kUpdate>(p, slice_max, s);
    }
}

// log2 of a block size the format allows (256, 512, 1024, 2048), else -1.
int qgrad_block_shift(int32_t block) {
    for (int sh = 8; sh <= 11; ++sh)
        if (block == (1 << sh)) return sh;
    return -1;
}

// The source checks shared by both entry points (no CUDA call).
int check_qsources(const int8_t* const* q_src, const float* const* scale_src, int32_t n_src,
                   int32_t block) {
    if (!q_src || !scale_src) return ZERO_EINVAL;
    if (n_src < 1) return ZERO_EINVAL;
    if (n_src > ZERO_MAX_SRC) return ZERO_ERANGE;
    if (qgrad_block_shift(block) < 0) return ZERO_EINVAL;
    for (int r = 0; r < n_src; ++r)
        if (!q_src[r] || !scale_src[r]) return ZERO_EINVAL;
    for (int r = 0; r < n_src; ++r)
        if (check_aligned(scale_src[r], 4)) return ZERO_EALIGN;
    return ZERO_OK;
}

int check_qsource_ptrs(const int8_t* const* q_src, const float* const* scale_src, int32_t n_src) {
    for (int r = 0; r < n_src; ++r)
        if (check_device_ptr(q_src[r]) || check_device_ptr(scale_src[r])) return ZERO_EINVAL;
    return ZERO_OK;
}

// The launches of a call over [begin, end): one over all owners' slices when
// the range is whole shards and every slice takes the vector kernel, else one
// per owner whose slice meets the range.  `place` sets the target pointers of a
// launch starting at flat `lo` and returns whether they allow the vector kernel.
template <bool kUpdate, bool kQ8, class Place>
int qgrad_run(const zero_layout_t* L, const int8_t* const* q_src, const float* const* scale_src,
              int32_t n_src, int32_t block, int64_t begin, int64_t end, QGradParams base,
              Place place, cudaStream_t s) {
    const int64_t S = L->shard;
    const int64_t nb = (S + block - 1) / block;
    base.n_src = n_src;
    base.block_shift = qgrad_block_shift(block);
    base.owners = 0;
    base.v8 = 0;
    base.o_first = 0;
    base.begin = base.end = base.S = base.nb = 0;
    for (int r = n_src; r < ZERO_MAX_SRC; ++r) {
        base.q[r] = nullptr;
        base.scale[r] = nullptr;
    }
    // whether the state (update) or destination (accumulation) of the element at
    // offset off from q's pointers starts on a 32-byte boundary
    auto a32 = [](const float* ptr, int64_t off) {
        return ptr != nullptr && ((reinterpret_cast<uintptr_t>(ptr) + (uintptr_t)off * 4u) & 31u) == 0;
    };
    auto v8_ok = [&](const QGradParams& q, int64_t off) {
        return kUpdate ? a32(q.w, off) && a32(q.m, off) && a32(q.v, off) : a32(q.dst, off);
    };
    // whether every source's slice of owner o starts on a 16-byte boundary (the
    // bulk copies of the warp-specialized kernel)
    auto slice_aligned16 = [&](int64_t o) {
        const int64_t lo = begin > o * S ? begin : o * S;
        for (int r = 0; r < n_src; ++r)
            if (!aligned16(q_src[r] + lo)) return false;
        return true;
    };
    // owner o's launch parameters and whether its slice takes the vector kernel
    auto owner_params = [&](int64_t o, QGradParams& p) {
        const int64_t lo = begin > o * S ? begin : o * S;
        const int64_t hi = end < (o + 1) * S ? end : (o + 1) * S;
        p = base;
        p.n = hi - lo;
        p.k0 = lo - o * S;
        bool vec = (p.k0 & 7) == 0;
        for (int r = 0; r < n_src; ++r) {
            p.q[r] = q_src[r] + lo;
            p.scale[r] = scale_src[r] + o * nb;
            vec = vec && (reinterpret_cast<uintptr_t>(p.q[r]) & 7u) == 0;
        }
        return place(p, lo) && vec;
    };
    const int64_t o_first = begin / S;
    const int64_t o_end = (end + S - 1) / S;               // owners o_first .. o_end - 1 meet the range
    bool all_vec = true, all_ws = true;
    int64_t slice_max = 0;
    QGradParams p;
    for (int64_t o = o_first; o < o_end; ++o) {
        all_vec = owner_params(o, p) && all_vec;
        all_ws = all_ws && slice_aligned16(o);
        slice_max = p.n > slice_max ? p.n : slice_max;
    }
    // Whole shards only: the owners share the grid's CTAs evenly, so slices of
    // unequal length would leave the CTAs of the short ones idle (measured:
    // -10 % on 5e8-element buckets over three owners, +4 to +11 % on the
    // per-unit calls over whole shards).
    const bool whole = begin % S == 0 && end % S == 0;
    // One stream over the whole range when every owner boundary lies on the
    // range's 8-element vector grid: a bucket that cuts shards is one launch
    // instead of one per owner (measured on GPT-2-XL shapes: 6466 against 6347
    // GB/s for the update).  Calls over whole shards keep the blockIdx.y grid
    // below, which measured faster than one stream for them (accumulation 6279
    // against 6075 GB/s; splitting the stream into equal blockIdx.y pieces did
    // not help either).
    const bool flat_grid = S % 8 == 0 && begin % 8 == 0;
    if (all_vec && flat_grid && o_end - o_first > 1 && (ZGB_QGRAD_FLAT == 2 || (ZGB_QGRAD_FLAT == 1 && !whole))) {
        p = base;
        p.owners = -1;
        p.o_first = (int32_t)o_first;
        p.begin = begin;
        p.end = end;
        p.S = S;
        p.nb = nb;
        p.n = end - begin;
        p.k0 = 0;
        for (int r = 0; r < n_src; ++r) {
            p.q[r] = q_src[r] + begin;
            p.scale[r] = scale_src[r];
        }
        (void)place(p, begin);
        p.v8 = qgrad_v8<kUpdate, kQ8>() && v8_ok(p, 0);
        return launch_qgrad<kUpdate, kQ8>(p, true, false, p.n, s);
    }
    if (ZGB_QGRAD_MULTI && whole && all_vec && o_end - o_first > 1 && o_end - o_first <= 65535) {
        // one launch, blockIdx.y = owner: every pointer at `begin`, the scales at their start
        p = base;
        p.owners = (int32_t)(o_end - o_first);
        p.o_first = (int32_t)o_first;
        p.begin = begin;
        p.end = end;
        p.S = S;
        p.nb = nb;
        p.n = p.k0 = 0;
        for (int r = 0; r < n_src; ++r) {
            p.q[r] = q_src[r] + begin;
            p.scale[r] = scale_src[r];
        }
        (void)place(p, begin);
        p.v8 = qgrad_v8<kUpdate, kQ8>();
        for (int64_t o = o_first; o < o_end; ++o)
            p.v8 = p.v8 && v8_ok(p, (begin > o * S ? begin : o * S) - begin);
        return launch_qgrad<kUpdate, kQ8>(p, true, all_ws, slice_max, s);
    }
    for (int64_t o = o_first; o < o_end; ++o) {
        const bool vec = owner_params(o, p);
        p.v8 = qgrad_v8<kUpdate, kQ8>() && v8_ok(p, 0);
        const int rc = launch_qgrad<kUpdate, kQ8>(p, vec, slice_aligned16(o), p.n, s);
        if (rc) return rc;
    }
    return ZERO_OK;
}

}  // namespace zgb

namespace zgb {

// The update from 8-bit gradients, with a bf16 output (out_bf16, out_mode) or
// the 8-bit output (q8: codes like the state, a scale per 256 elements).
int qgrad_update(const zero_layout_t* L, const int8_t* const* q_src, const float* const* scale_src,
                 int32_t n_src, int32_t block, float divisor, int32_t rank_begin, int32_t rank_end,
                 int64_t begin, int64_t end, float* master, float* m, float* v, uint16_t* out_bf16,
                 int32_t out_mode, int8_t* q_out, float* scales_out, const zero_adamw_t* hp,
                 void* stream) {
    int rc = check_qsources(q_src, scale_src, n_src, block);
    if (rc) return rc;
    if (q_out) {
        if (!L || !scales_out) return ZERO_EINVAL;
        if (L->shard % 256 != 0 || begin % 256 != 0 || end % 256 != 0) return ZERO_EINVAL;
        if (check_aligned(scales_out, 4)) return ZERO_EALIGN;
    }
    UpdateTarget t;
    if ((rc = prepare_target(L, rank_begin, rank_end, begin, end, master, m, v, out_bf16, out_mode,
                             q_out != nullptr, &t)))
        return rc;
    QGradParams base;
    if ((rc = make_scalars(hp, divisor, &base.h))) return rc;
    if (end == begin) return ZERO_OK;
    if ((rc = check_qsource_ptrs(q_src, scale_src, n_src))) return rc;
    if ((rc = check_target_ptrs(t))) return rc;
    if (q_out && (check_device_ptr(q_out) || check_device_ptr(scales_out))) return ZERO_EINVAL;
    base.dst = nullptr;
    base.first = 0;
    base.out = nullptr;
    base.qout = nullptr;
    base.qoscale = nullptr;
    const int64_t own_lo = (int64_t)rank_begin * L->shard;
    auto place = [&](QGradParams& p, int64_t lo) {
        const int64_t off = lo - begin;
        p.w = t.w + off;
        p.m = t.m + off;
        p.v = t.v + off;
        bool ok = aligned16(p.w) && aligned16(p.m) && aligned16(p.v);
        if (q_out) {
            p.qout = q_out + (lo - own_lo);              // lo - own_lo is a multiple of 256
            p.qoscale = scales_out + (lo - own_lo) / 256;
            ok = ok && aligned16(p.qout);
        } else {
            p.out = t.out + off;
            ok = ok && aligned16(p.out);
        }
        return ok;
    };
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return q_out ? qgrad_run<true, true>(L, q_src, scale_src, n_src, block, begin, end, base, place, s)
                 : qgrad_run<true, false>(L, q_src, scale_src, n_src, block, begin, end, base, place, s);
}

}  // namespace zgb

extern "C" int zero_reduce_scatter_adamw_int8(const zero_layout_t* L, const int8_t* const* q_src,
                                              const float* const* scale_src, int32_t n_src,
                                              int32_t block, float divisor, int32_t rank_begin,
                                              int32_t rank_end, int64_t begin, int64_t end,
                                              float* master, float* m, float* v, uint16_t* out_bf16,
                                              int32_t out_mode, const zero_adamw_t* hp, void* stream) {
    if (out_mode == zgb::ZERO_OUT_NONE) return ZERO_EINVAL;
    return zgb::qgrad_update(L, q_src, scale_src, n_src, block, divisor, rank_begin, rank_end, begin,
                             end, master, m, v, out_bf16, out_mode, nullptr, nullptr, hp, stream);
}

extern "C" int zero_reduce_scatter_adamw_int8_q8(const zero_layout_t* L, const int8_t* const* q_src,
                                                 const float* const* scale_src, int32_t n_src,
                                                 int32_t block, float divisor, int32_t rank_begin,
                                                 int32_t rank_end, int64_t begin, int64_t end,
                                                 float* master, float* m, float* v, int8_t* q_out,
                                                 float* scales_out, int32_t out_block,
                                                 const zero_adamw_t* hp, void* stream) {
    if (!q_out || out_block != 256) return ZERO_EINVAL;
    return zgb::qgrad_update(L, q_src, scale_src, n_src, block, divisor, rank_begin, rank_end, begin,
                             end, master, m, v, nullptr, zgb::ZERO_OUT_NONE, q_out, scales_out, hp,
                             stream);
}

extern "C" int zero_accumulate_int8(const zero_layout_t* L, const int8_t* const* q_src,
                                    const float* const* scale_src, int32_t n_src, int32_t block,
                                    float* dst, int64_t dst_base, int64_t begin, int64_t end,
                                    int32_t first, void* stream) {
    using namespace zgb;
    if (!L || !dst) return ZERO_EINVAL;
    int rc = check_qsources(q_src, scale_src, n_src, block);
    if (rc) return rc;
    if (!layout_shape_ok(L))
        return ZERO_EINVAL;
    if (begin < 0 || end > L->padded_n || begin > end) return ZERO_EINVAL;
    if (dst_base > begin) return ZERO_EINVAL;
    if (check_aligned(dst, 4)) return ZERO_EALIGN;
    if (end == begin) return ZERO_OK;
    if ((rc = check_qsource_ptrs(q_src, scale_src, n_src))) return rc;
    if (check_device_ptr(dst)) return ZERO_EINVAL;
    QGradParams base;
    base.w = base.m = base.v = nullptr;
    base.out = nullptr;
    base.qout = nullptr;
    base.qoscale = nullptr;
    base.first = first ? 1 : 0;
    base.h = AdamwScalars{};
    auto place = [&](QGradParams& p, int64_t lo) {
        p.dst = dst + (lo - dst_base);
        return aligned16(p.dst);
    };
    return qgrad_run<false, false>(L, q_src, scale_src, n_src, block, begin, end, base, place,
                            static_cast<cudaStream_t>(stream));
}

