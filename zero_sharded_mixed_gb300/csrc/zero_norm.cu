// Squared global norm of the mean gradient, for clipping by the global norm
// ("DeepSpeed ZeRO", "The configuration file" and "ZeRO Optimizer, in depth",
// "Running it with DeepSpeed": gradient_clipping 1.0), sm_103a.
//
// For every flat i in [begin, end) the mean gradient g_i is formed exactly as
// the fused update forms it (fp32 sum over sources in ascending order from
// +0.0f, one IEEE division -- for a power-of-two divisor the multiply by its
// exact reciprocal, which rounds the same real number), and g_i^2 is added to
// the thread's running sum.
// fp64 arithmetic is slow on this GPU (a few per element would bound the pass
// below the HBM rate), so the thread's sum is kept as an unevaluated pair of
// fp32 values (hi, lo): the square is split exactly into p + e by the FMA
// two-product (Dekker; Ogita, Rump and Oishi, "Accurate sum and dot product",
// 2005) and added with Knuth's two-sum, whose rounding error goes into lo.
// The pair carries about 48 significant bits; squares outside the range where
// that split is exact (|g| < 2^-50 or >= 2^60) go to a plain fp64 sum instead.
// Pass 1 (one streaming kernel, 2 bytes per bf16 source per element): each
// thread sums its elements in order, widens its pair to fp64, each CTA reduces
// its threads in a fixed tree and writes one fp64 partial into the caller's
// workspace.  Pass 2
// (one CTA): the partials are summed in a fixed tree and the total is written
// to (or added to) *norm_sq in device memory, where the clipped update reads
// it -- nothing returns to the host.  For a given GPU and range the grid, and
// so the summation order, is fixed: results are reproducible run to run.
#include <atomic>
#include <cmath>

#include "zero_common.cuh"

namespace zgb {

#ifndef ZGB_NORM_POW2
#define ZGB_NORM_POW2 1      // 1: a power-of-two divisor is applied as a multiply by its exact
                             // reciprocal (the same correctly rounded value as the division;
                             // measured +6.6 % on the 8-source pass, 7129 against 6689 GB/s)
#endif
#ifndef ZGB_NORM_U
#define ZGB_NORM_U 1         // vectors per thread and pass (2: vi and vi + stride together;
                             // 128 registers, within noise of 1)
#endif

constexpr int kMaxCtasPerSm = 2048 / kThreads;   // upper bound on resident CTAs of kThreads

struct NormParams {
    const void* src[ZERO_MAX_SRC];  // offset to the first element of the range
    int64_t n;
    int32_t n_src;
    float divisor;
    float inv_divisor;              // 1/divisor when divisor is a power of two, else 0
    double* partials;               // one per CTA
};

__device__ __forceinline__ float norm_mean(float s, const NormParams& p) {
    if (ZGB_NORM_POW2 && p.inv_divisor != 0.0f) return __fmul_rn(s, p.inv_divisor);
    return __fdiv_rn(s, p.divisor);
}

template <bool kBf16>
__device__ __forceinline__ float mean_at(const NormParams& p, int64_t i) {
    float s = 0.0f;
    for (int r = 0; r < p.n_src; ++r)
        s = __fadd_rn(s, kBf16 ? bf16_one(static_cast<const uint16_t*>(p.src[r])[i])
                               : static_cast<const float*>(p.src[r])[i]);
    return norm_mean(s, p);
}

// A thread's running sum of squares: (hi + lo) in fp32 pairs plus an fp64 sum
// for squares outside the range where the fp32 split is exact.
struct SquareSum {
    float hi = 0.0f, lo = 0.0f;
    double wide = 0.0;

    __device__ __forceinline__ void add(float g) {
        const float a = fabsf(g);
        if (a >= 0x1p-50f && a < 0x1p+60f) {
            const float p = __fmul_rn(g, g);
            const float e = __fmaf_rn(g, g, -p);                 // g*g = p + e exactly
            const float t = __fadd_rn(hi, p);                    // two-sum of hi and p
            const float bp = __fsub_rn(t, hi);
            const float err = __fadd_rn(__fsub_rn(hi, __fsub_rn(t, bp)), __fsub_rn(p, bp));
            hi = t;
            lo = __fadd_rn(lo, __fadd_rn(err, e));
        } else if (a != 0.0f) {
            const double d = (double)g;
            wide = __dadd_rn(wide, __dmul_rn(d, d));
        }
    }

    __device__ __forceinline__ double total() const {
        return __dadd_rn(__dadd_rn((double)hi, (double)lo), wide);
    }
};

// Fixed-order CTA reduction of one fp64 value per thread; thread 0 gets the total.
__device__ __forceinline__ double cta_sum(double x) {
    __shared__ double warp_sums[kThreads / 32];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_down_sync(0xffffffffu, x, off);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) warp_sums[warp] = x;
    __syncthreads();
    double t = 0.0;
    if (warp == 0) {
        t = lane < kThreads / 32 ? warp_sums[lane] : 0.0;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) t += __shfl_down_sync(0xffffffffu, t, off);
    }
    return t;
}

// One vector's sources: R 16-byte loads of bf16, or 2R of fp32.
template <bool kBf16, int R>
struct NormVec {
    uint4 u[kBf16 ? R : 1];
    float4 f[kBf16 ? 1 : 2 * R];
};

template <bool kBf16, int R>
__device__ __forceinline__ void norm_load(const NormParams& p, int64_t e, NormVec<kBf16, R>& x) {
#pragma unroll
    for (int r = 0; r < R; ++r) {
        if constexpr (kBf16) {
            x.u[r] = ld_stream_u4(static_cast<const uint16_t*>(p.src[r]) + e);
        } else {
            x.f[2 * r] = ld_stream_f4(static_cast<const float*>(p.src[r]) + e);
            x.f[2 * r + 1] = ld_stream_f4(static_cast<const float*>(p.src[r]) + e + 4);
        }
    }
}

// The vector's 8 means (sources summed in ascending order from +0.0f) and
// their squares into the thread's sum.
template <bool kBf16, int R>
__device__ __forceinline__ void norm_add(const NormParams& p, const NormVec<kBf16, R>& x, SquareSum& acc) {
    float s[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) s[j] = 0.0f;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        if constexpr (kBf16) {
            const uint32_t w4[4] = {x.u[r].x, x.u[r].y, x.u[r].z, x.u[r].w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                s[2 * k] = __fadd_rn(s[2 * k], bf16_lo(w4[k]));
                s[2 * k + 1] = __fadd_rn(s[2 * k + 1], bf16_hi(w4[k]));
            }
        } else {
            const float4 lo = x.f[2 * r], hi = x.f[2 * r + 1];
            s[0] = __fadd_rn(s[0], lo.x); s[1] = __fadd_rn(s[1], lo.y);
            s[2] = __fadd_rn(s[2], lo.z); s[3] = __fadd_rn(s[3], lo.w);
            s[4] = __fadd_rn(s[4], hi.x); s[5] = __fadd_rn(s[5], hi.y);
            s[6] = __fadd_rn(s[6], hi.z); s[7] = __fadd_rn(s[7], hi.w);
        }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) acc.add(norm_mean(s[j], p));
}

template <bool kBf16, int R>
__global__ void __launch_bounds__(kThreads) norm_partial_kernel(const __grid_constant__ NormParams p) {
    const int64_t tid = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    SquareSum acc;
    if constexpr (R > 0) {
        const int64_t nv = p.n >> 3;
        // U vectors per pass: vi, vi + stride, ... (the same elements in the same
        // order as one vector per pass)
        constexpr int U = ZGB_NORM_U;
        for (int64_t vi = tid; vi < nv; vi += (int64_t)U * stride) {
            NormVec<kBf16, R> x[U];
            bool ok[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                ok[u] = vi + u * stride < nv;
                if (ok[u]) norm_load<kBf16, R>(p, (vi + u * stride) * 8, x[u]);
            }
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (ok[u]) norm_add<kBf16, R>(p, x[u], acc);
        }
        const int64_t tail = p.n - (nv << 3);
        if (tid < tail) acc.add(mean_at<kBf16>(p, (nv << 3) + tid));
    } else {
        for (int64_t i = tid; i < p.n; i += stride) acc.add(mean_at<kBf16>(p, i));
    }
    const double total = cta_sum(acc.total());
    if (threadIdx.x == 0) p.partials[blockIdx.x] = total;
}

__global__ void __launch_bounds__(kThreads)
norm_finalize_kernel(const double* partials, int n_partials, double* norm_sq, int accumulate) {
    double acc = 0.0;
    for (int i = threadIdx.x; i < n_partials; i += kThreads) acc = __dadd_rn(acc, partials[i]);
    const double total = cta_sum(acc);
    if (threadIdx.x == 0) *norm_sq = accumulate ? __dadd_rn(*norm_sq, total) : total;
}

// CTAs the partial kernel may launch on this device (one partial each).
int64_t norm_partials_capacity() { return (int64_t)sm_count() * kMaxCtasPerSm; }

template <bool kBf16, int R>
int launch_norm(const NormParams& p, bool vec, double* norm_sq, int accumulate, cudaStream_t s) {
    const int occupancy = ctas_per_sm((const void*)norm_partial_kernel<kBf16, R>, kThreads, 0);
    const int64_t resident = (int64_t)sm_count() * (occupancy < kMaxCtasPerSm ? occupancy : kMaxCtasPerSm);
    const unsigned grid = grid_for(vec ? (p.n >> 3) : p.n, kThreads, resident);
    norm_partial_kernel<kBf16, R><<<grid, kThreads, 0, s>>>(p);
    int rc = launch_status();
    if (rc) return rc;
    norm_finalize_kernel<<<1, kThreads, 0, s>>>(p.partials, (int)grid, norm_sq, accumulate);
    return launch_status();
}

template <bool kBf16>
int dispatch_norm(const NormParams& p, bool vec, double* norm_sq, int accumulate, cudaStream_t s) {
    if (!vec) return launch_norm<kBf16, 0>(p, false, norm_sq, accumulate, s);
    switch (p.n_src) {
        case 1: return launch_norm<kBf16, 1>(p, true, norm_sq, accumulate, s);
        case 2: return launch_norm<kBf16, 2>(p, true, norm_sq, accumulate, s);
        case 4: return launch_norm<kBf16, 4>(p, true, norm_sq, accumulate, s);
        case 8: return launch_norm<kBf16, 8>(p, true, norm_sq, accumulate, s);
        default: return launch_norm<kBf16, 0>(p, false, norm_sq, accumulate, s);
    }
}

// The body of zero_grad_norm_sq: argument checks, then the two launches.
int grad_norm_sq(const zero_layout_t* L, const void* const* src, int32_t n_src, int32_t src_dtype,
                 int64_t src_base, float divisor, int64_t begin, int64_t end, double* partials,
                 int64_t partials_len, double* norm_sq, int32_t accumulate, void* stream) {
    if (!L || !src || !norm_sq) return ZERO_EINVAL;
    if (n_src < 1) return ZERO_EINVAL;
    if (n_src > ZERO_MAX_SRC) return ZERO_ERANGE;
    if (src_dtype != ZERO_BF16 && src_dtype != ZERO_F32) return ZERO_EINVAL;
    if (!layout_shape_ok(L)) return ZERO_EINVAL;
    if (begin < 0 || end > L->padded_n || begin > end || src_base > begin) return ZERO_EINVAL;
    if (!(divisor > 0.0f) || !(divisor < 3.4e38f)) return ZERO_EINVAL;
    for (int r = 0; r < n_src; ++r)
        if (!src[r]) return ZERO_EINVAL;
    const int esize = src_dtype == ZERO_BF16 ? 2 : 4;
    for (int r = 0; r < n_src; ++r)
        if (check_aligned(src[r], esize)) return ZERO_EALIGN;
    if (check_aligned(norm_sq, 8) || check_aligned(partials, 8)) return ZERO_EALIGN;
    for (int r = 0; r < n_src; ++r)
        if (check_device_ptr(src[r])) return ZERO_EINVAL;
    if (check_device_ptr(norm_sq)) return ZERO_EINVAL;
    if (!partials || partials_len < norm_partials_capacity()) return ZERO_ERANGE;
    if (check_device_ptr(partials)) return ZERO_EINVAL;
    NormParams p;
    bool vec = true;
    for (int r = 0; r < ZERO_MAX_SRC; ++r) p.src[r] = nullptr;
    for (int r = 0; r < n_src; ++r) {
        p.src[r] = static_cast<const char*>(src[r]) + (begin - src_base) * esize;
        vec = vec && aligned16(p.src[r]);
    }
    p.n = end - begin;
    p.n_src = n_src;
    p.divisor = divisor;
    int e2 = 0;
    const float mant = std::frexp(divisor, &e2);          // divisor = mant * 2^e2, mant in [0.5, 1)
    p.inv_divisor = (mant == 0.5f && e2 >= -125 && e2 <= 127) ? std::ldexp(1.0f, 1 - e2) : 0.0f;
    p.partials = partials;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return src_dtype == ZERO_BF16 ? dispatch_norm<true>(p, vec, norm_sq, accumulate ? 1 : 0, s)
                                  : dispatch_norm<false>(p, vec, norm_sq, accumulate ? 1 : 0, s);
}

}  // namespace zgb

extern "C" int zero_grad_norm_workspace(int64_t* bytes) {
    if (!bytes) return ZERO_EINVAL;
    *bytes = zgb::norm_partials_capacity() * (int64_t)sizeof(double);
    return ZERO_OK;
}

extern "C" int zero_grad_norm_sq(const zero_layout_t* L, const void* const* src, int32_t n_src,
                                 int32_t src_dtype, int64_t src_base, float divisor, int64_t begin,
                                 int64_t end, void* workspace, int64_t workspace_bytes,
                                 double* norm_sq, int32_t accumulate, void* stream) {
    using namespace zgb;
    return grad_norm_sq(L, src, n_src, src_dtype, src_base, divisor, begin, end,
                        static_cast<double*>(workspace), workspace_bytes / (int64_t)sizeof(double),
                        norm_sq, accumulate, stream);
}

// ---------------------------------------------------------------------------
// zero_grad_norm_sq_static: the same computation with its partial sums in a
// fixed array of device memory that belongs to this library, for callers that
// cannot hand it a workspace.
// ---------------------------------------------------------------------------

namespace zgb {

// Capacity of the library-owned partials: one fp64 per CTA of the partial
// pass, which launches at most (SMs x kMaxCtasPerSm) CTAs.  Sized for GPUs of
// up to 512 SMs whatever the build's CTA size: 4096 doubles (32 KiB) at the
// default 256 threads, 16384 (128 KiB) at 64.  Held by every GPU that loads
// the library until the process exits.
constexpr int64_t kStaticMaxSms = 512;
constexpr int64_t kStaticPartials = kStaticMaxSms * kMaxCtasPerSm;
static __device__ __align__(256) double g_static_partials[kStaticPartials];

namespace {
constexpr int kMaxStaticDevices = 64;
std::atomic<double*> g_static_partials_addr[kMaxStaticDevices];
}  // namespace

// The device address of g_static_partials on the current device, looked up
// once per device (cudaGetSymbolAddress with that device current) and cached;
// refresh = true looks it up again (after the device's context was replaced).
int static_partials(double** out, bool refresh) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
        (void)cudaGetLastError();
        return ZERO_ECUDA;
    }
    if (dev >= kMaxStaticDevices) return ZERO_ERANGE;
    double* p = refresh ? nullptr : g_static_partials_addr[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        void* addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_static_partials) != cudaSuccess || addr == nullptr) {
            (void)cudaGetLastError();
            return ZERO_ECUDA;
        }
        p = static_cast<double*>(addr);
        g_static_partials_addr[dev].store(p, std::memory_order_release);
    }
    *out = p;
    return ZERO_OK;
}

}  // namespace zgb

extern "C" int zero_grad_norm_sq_static(const zero_layout_t* L, const void* const* src,
                                        int32_t n_src, int32_t src_dtype, int64_t src_base,
                                        float divisor, int64_t begin, int64_t end, double* norm_sq,
                                        int32_t accumulate, void* stream) {
    using namespace zgb;
    if (!L || !src || !norm_sq) return ZERO_EINVAL;
    if (norm_partials_capacity() > kStaticPartials) return ZERO_ERANGE;   // more SMs than it holds
    double* partials = nullptr;
    int rc = static_partials(&partials, false);
    if (rc) return rc;
    // A cached address that is no longer device memory of this device means the
    // context it came from was destroyed (cudaDeviceReset): look it up again.
    if (check_device_ptr(partials) && (rc = static_partials(&partials, true))) return rc;
    // Every partial the finalize pass reads is written by the partial pass of
    // the same call, so nothing in the array needs clearing between calls.
    return grad_norm_sq(L, src, n_src, src_dtype, src_base, divisor, begin, end, partials,
                        kStaticPartials, norm_sq, accumulate, stream);
}
