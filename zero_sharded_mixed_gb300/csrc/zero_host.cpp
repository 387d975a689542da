// Host-only parts of libzero_gb300.so: layout, ranges, status strings and the
// memory / communication accounting.  No CUDA call is made here.
#include <cmath>
#include <cstdint>
#include <limits>

#include "zero_gb300.h"

namespace {

constexpr int64_t kMaxElems = std::numeric_limits<int64_t>::max() / 8;

// a + b and a * b for non-negative operands, false when past kMaxElems
bool add_ok(int64_t a, int64_t b, int64_t* r) {
    if (a > kMaxElems - b) return false;
    *r = a + b;
    return true;
}
bool mul_ok(int64_t a, int64_t b, int64_t* r) {
    if (a != 0 && b > kMaxElems / a) return false;
    *r = a * b;
    return true;
}
int64_t ceil_div(int64_t a, int64_t b) { return a == 0 ? 0 : 1 + (a - 1) / b; }

}  // namespace

extern "C" int zero_layout(const int64_t* numel, int32_t n_tensors, int32_t n_dp, int64_t align,
                           int64_t bucket_elems, int64_t* offsets_out, zero_layout_t* out) {
    if (out == nullptr || n_tensors < 0 || n_dp < 1 || align < 1 || bucket_elems < 1)
        return ZERO_EINVAL;
    if (n_tensors > 0 && numel == nullptr) return ZERO_EINVAL;
    int64_t n = 0;
    for (int32_t t = 0; t < n_tensors; ++t) {
        if (numel[t] < 0) return ZERO_EINVAL;
        if (offsets_out) offsets_out[t] = n;
        if (!add_ok(n, numel[t], &n)) return ZERO_ERANGE;
    }
    // S: the smallest multiple of align whose n_dp copies hold all n elements
    int64_t shard = 0;
    if (!mul_ok(ceil_div(ceil_div(n, n_dp), align), align, &shard)) return ZERO_ERANGE;
    int64_t padded = 0;
    if (!mul_ok(shard, n_dp, &padded)) return ZERO_ERANGE;
    int64_t bucket = 0;
    if (!mul_ok(ceil_div(bucket_elems, align), align, &bucket)) return ZERO_ERANGE;
    zero_layout_t L;
    L.n = n;
    L.padded_n = padded;
    L.shard = shard;
    L.align = align;
    L.bucket = bucket;
    L.n_buckets = ceil_div(padded, bucket);
    L.n_dp = n_dp;
    L.reserved = 0;
    *out = L;
    return ZERO_OK;
}

extern "C" int zero_bucket_range(const zero_layout_t* L, int64_t b, int64_t* begin, int64_t* end) {
    if (!L || !begin || !end || b < 0 || b >= L->n_buckets || L->bucket < 1) return ZERO_EINVAL;
    int64_t lo = 0, e = 0;                  // a caller's layout: no product past kMaxElems
    if (!mul_ok(b, L->bucket, &lo) || !add_ok(lo, L->bucket, &e)) return ZERO_EINVAL;
    *begin = lo;
    *end = e < L->padded_n ? e : L->padded_n;
    return ZERO_OK;
}

extern "C" int zero_shard_range(const zero_layout_t* L, int32_t rank, int64_t* begin, int64_t* end,
                                int64_t* valid_end) {
    if (!L || !begin || !end || rank < 0 || rank >= L->n_dp || L->shard < 0) return ZERO_EINVAL;
    int64_t b = 0, e = 0;                   // a caller's layout: no product past kMaxElems
    if (!mul_ok(rank, L->shard, &b) || !add_ok(b, L->shard, &e)) return ZERO_EINVAL;
    *begin = b;
    *end = e;
    if (valid_end) *valid_end = L->n < b ? b : (L->n < e ? L->n : e);
    return ZERO_OK;
}

extern "C" const char* zero_strerror(int code) {
    switch (code) {
        case ZERO_OK: return "ok";
        case ZERO_EINVAL: return "invalid argument";
        case ZERO_EALIGN: return "misaligned pointer";
        case ZERO_ERANGE: return "size out of range";
        case ZERO_ECUDA: return "CUDA runtime error";
        case ZERO_ETIMEOUT: return "device-side wait timed out";
        case ZERO_EIO: return "checkpoint file I/O error";
        case ZERO_ECORRUPT: return "checkpoint file corrupt (magic, version or CRC)";
        default: return "unknown status code";
    }
}

extern "C" int zero_memory_bytes(double n, int32_t n_dp, int32_t stage, double k_bytes, double* out) {
    if (!out || n_dp < 1 || n < 0 || stage < 0 || stage > 3 || !(k_bytes >= 0)) return ZERO_EINVAL;
    // one more kind of state moves under 1/n_dp at each stage
    double shards = (double)n_dp;
    double weights = 2.0 * n / (stage >= 3 ? shards : 1.0);
    double grads = 2.0 * n / (stage >= 2 ? shards : 1.0);
    double optim = k_bytes * n / (stage >= 1 ? shards : 1.0);
    *out = weights + grads + optim;
    return ZERO_OK;
}

extern "C" int zero_comm_bytes(double n, int32_t n_dp, int32_t stage, double param_bytes,
                               double grad_bytes, double* out) {
    if (!out || n_dp < 1 || n < 0 || stage < 0 || stage > 3 || !(param_bytes >= 0) ||
        !(grad_bytes >= 0))
        return ZERO_EINVAL;
    // a ring reduce-scatter or all-gather of n elements sends (n_dp-1)/n_dp * n per GPU
    double ring = (double)(n_dp - 1) / (double)n_dp * n;
    double gather_passes = stage == 0 ? 0.0 : (stage == 3 ? 2.0 : 1.0);
    double grad_passes = stage == 0 ? 2.0 : 1.0;   // all-reduce = reduce-scatter + all-gather
    *out = ring * (grad_passes * grad_bytes + gather_passes * param_bytes);
    return ZERO_OK;
}

extern "C" int zero_lr_warmup_decay(int64_t t, double min_lr, double max_lr, int64_t warmup_steps,
                                    int64_t total_steps, float* lr_out) {
    if (!lr_out || t < 1 || warmup_steps < 0 || total_steps <= warmup_steps) return ZERO_EINVAL;
    if (!std::isfinite(min_lr) || !std::isfinite(max_lr) || min_lr < 0 || max_lr < 0) return ZERO_EINVAL;
    const int64_t k = t - 1;                         // schedule steps taken before step t
    double lr = 0.0;
    if (k < warmup_steps)
        lr = min_lr + (max_lr - min_lr) * ((double)k / (double)warmup_steps);
    else if (k < total_steps)
        lr = max_lr * ((double)(total_steps - k) / (double)(total_steps - warmup_steps));
    *lr_out = (float)lr;
    return ZERO_OK;
}
