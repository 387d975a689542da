/*
 * zero_gb300.h -- C ABI of libzero_gb300.so: the ZeRO stage-1/2/3 sharded
 * mixed-precision optimizer step on one GB300 (sm_103a).
 *
 * The n_dp data-parallel ranks are simulated as separate buffers in the one
 * GPU's memory: rank r's full local gradient is its own buffer, rank o's shard
 * of the fp32 master weights and Adam moments is its own range, and a
 * "collective" is a kernel reading and writing those buffers.
 *
 * Conventions for every call:
 *  - Return value: 0 (ZERO_OK) or a negative ZERO_E* code; zero_strerror()
 *    names it.  A call that returns an error has enqueued nothing.
 *  - Memory: the caller owns every buffer.  The library never allocates or
 *    frees device memory and never synchronizes, except zero_status_check().
 *    Every buffer argument must be device memory of the current device
 *    (checked: host or other-device pointers give ZERO_EINVAL; the gradient
 *    sources of zero_reduce_scatter_adamw may also be pinned host memory, and
 *    the layout, schedule-table and checkpoint calls work on host memory) and at least
 *    element-aligned (2 bytes for bf16, 4 for fp32; else ZERO_EALIGN).  When all
 *    the pointers of a call, after offsetting to the start of the range, are
 *    16-byte aligned the kernels move 128-bit vectors; otherwise the same
 *    kernels run element by element (still on the GPU).  The library cannot see
 *    buffer lengths: extents stated below are the caller's responsibility (the
 *    Python binding checks them against the tensors it is given).
 *  - bf16 values are passed as uint16_t bit patterns.
 *  - Streams: `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *    default stream).  Work is enqueued on it asynchronously.
 *  - Pointer arrays (`src`, `shards`) are HOST arrays of device pointers.
 *  - Layouts: a zero_layout_t passed in must have the shape zero_layout()
 *    gives (n_dp >= 1, shard >= 0, padded_n = shard * n_dp, at most
 *    2^63 / 8 elements); a hand-made struct outside that shape gives
 *    ZERO_EINVAL, checked before any product of its fields is formed.
 *
 * Notation ("ZeRO and FSDP", section "The idea, one stage at a time"): all
 * parameters are flattened into one vector of N elements and cut into n_dp
 * equal contiguous shards; rank r owns shard r.  Here the shard length is
 * S = round_up(ceil(N / n_dp), align), the padded length P = n_dp * S, and the
 * padding tail [N, P) holds zeros in every buffer.
 */
#ifndef ZERO_GB300_H
#define ZERO_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
enum {
    ZERO_OK = 0,
    ZERO_EINVAL = -1,   /* an argument is out of its domain (null, range, mode, pointer kind) */
    ZERO_EALIGN = -2,   /* a pointer is not aligned to its element size */
    ZERO_ERANGE = -3,   /* a size does not fit (int64 overflow, too many sources), or a
                           step schedule was advanced past its table */
    ZERO_ECUDA = -4,    /* the CUDA runtime reported an error (launch or earlier async fault) */
    ZERO_ETIMEOUT = -5, /* a bounded device-side wait gave up (zero_status_check) */
    ZERO_EIO = -6,      /* a checkpoint file could not be opened, written or read */
    ZERO_ECORRUPT = -7  /* a checkpoint file has a wrong magic, version or CRC */
};

/* ---- enums -------------------------------------------------------------- */
enum { ZERO_BF16 = 0, ZERO_F32 = 1 };                 /* source element type */
enum { ZERO_OUT_FULL = 0, ZERO_OUT_SHARD = 1 };       /* where the bf16 result goes */
enum { ZERO_ACC_LOCAL = 0, ZERO_ACC_REDUCE = 1 };     /* accumulation mode */

#define ZERO_MAX_SRC 64   /* most source buffers one call reads */

/* ---- structures --------------------------------------------------------- */

/* A flat layout (one model under ZeRO-1/2, or one unit under ZeRO-3). */
typedef struct {
    int64_t n;          /* N: real elements */
    int64_t padded_n;   /* P = n_dp * shard */
    int64_t shard;      /* S: elements per rank, a multiple of align */
    int64_t align;      /* a: shard alignment in elements */
    int64_t bucket;     /* bucket length in elements, a multiple of align */
    int64_t n_buckets;  /* ceil(P / bucket); 0 when P == 0 */
    int32_t n_dp;       /* number of (simulated) data-parallel ranks */
    int32_t reserved;   /* zero */
} zero_layout_t;

/* AdamW hyper-parameters for one step. */
typedef struct {
    float lr;
    float beta1;
    float beta2;
    float eps;
    float weight_decay;
    int32_t reserved;   /* zero */
    int64_t step;       /* t, starting at 1 */
    /* NULL, or a DEVICE pointer to 3 floats {lr, 1 - beta1^t, 1 - beta2^t} of the
     * current step, read by the kernels in place of lr and step (written by
     * zero_schedule_advance from a table of zero_schedule_fill): the step's
     * scalars then live in device memory, so that a captured CUDA graph of a
     * step can be replayed step after step.  4-byte aligned. */
    const float* sched;
} zero_adamw_t;

/* ---- layout --------------------------------------------------------------
 * "ZeRO and FSDP", "The idea, one stage at a time" (flatten into one vector,
 * n_dp equal contiguous shards, rank r owns shard r); "ZeRO Optimizer, in
 * depth", "Worked example" (reduce buckets of 5e8 elements by default).
 *
 * numel[n_tensors]: element counts in flattening order (tensors are laid end
 *   to end, no gaps).  align >= 1; bucket_elems >= 1 (rounded up to a multiple
 *   of align).  offsets_out (host, n_tensors entries, may be NULL) receives each
 *   tensor's flat offset.  out (host) receives the layout.
 * Errors: ZERO_EINVAL (n_dp < 1, align < 1, bucket_elems < 1, negative numel,
 *   null out / numel), ZERO_ERANGE (sizes overflow).  Host-only; no CUDA call. */
int zero_layout(const int64_t* numel, int32_t n_tensors, int32_t n_dp, int64_t align,
                int64_t bucket_elems, int64_t* offsets_out, zero_layout_t* out);

/* Bucket b covers the flat range [*begin, *end) = [b*bucket, min((b+1)*bucket, P)).
 * ZERO_EINVAL unless 0 <= b < n_buckets.  Host-only. */
int zero_bucket_range(const zero_layout_t* L, int64_t b, int64_t* begin, int64_t* end);

/* Rank r owns [*begin, *end) = [r*S, (r+1)*S); *valid_end = min(max(N, begin), end)
 * is where its real elements stop.  ZERO_EINVAL unless 0 <= r < n_dp.  Host-only. */
int zero_shard_range(const zero_layout_t* L, int32_t rank, int64_t* begin, int64_t* end,
                     int64_t* valid_end);

/* ---- the fused step ------------------------------------------------------
 * "ZeRO and FSDP", "The idea, one stage at a time" (stage 1: reduce-scatter so
 * rank r receives the averaged gradient of shard r, update the fp32 master
 * shard, cast to bf16, all-gather; stage 2: the same per gradient bucket as
 * it becomes ready) and exercise "A sharded Adam step" (Adam with bias
 * correction at step t); AdamW's decoupled weight decay per the optimizer
 * blocks of "DeepSpeed ZeRO", "The configuration file".
 *
 * For every flat index i in [begin, end):
 *   g      = (sum over r = 0..n_src-1 of src[r][i - src_base]) / divisor
 *            (fp32, ranks in ascending order from +0.0f, one IEEE division)
 *   m      = b1*m + (1-b1)*g;   v = b2*v + (1-b2)*g*g
 *   w      = w - (lr*wd)*w;     w = w - lr*((m/bc1) / (sqrt(v/bc2) + eps))
 *   out    = bf16 round-to-nearest-even of w
 * with bc1 = 1 - b1^t, bc2 = 1 - b2^t evaluated in fp64 on the host and
 * rounded to fp32, every other operation one IEEE fp32 rounding (no FMA).
 *
 * Indexing: rank_begin..rank_end-1 are the owners whose shards this call
 *   updates; [begin, end) must lie inside [rank_begin*S, rank_end*S).
 *   master/m/v point at rank_begin's shard; the state of flat index i is at
 *   [i - rank_begin*S] (the owned shards of consecutive ranks are contiguous).
 *   out_mode ZERO_OUT_FULL: out_bf16 is the full flat bf16 weight buffer of P
 *   elements and receives [i] -- the all-gather of stages 1 and 2.
 *   out_mode ZERO_OUT_SHARD: out_bf16 is laid out like master and receives
 *   [i - rank_begin*S] -- the stage-3 owner updating its own bf16 shard.
 *   src[r] (n_src of them, 1 <= n_src <= ZERO_MAX_SRC) is read at [i - src_base];
 *   src_dtype ZERO_BF16 (per-rank bf16 gradients) or ZERO_F32 (accumulated
 *   fp32 gradients).  src_base <= begin.  divisor > 0 and finite (n_dp for a
 *   mean over ranks, n_dp*K after K accumulated micro-batches).
 * Memory: master, m, v and out are device memory of the current device.  Each
 *   src[r] is device memory or pinned host memory that the device addresses
 *   at the same pointer (page-locked, mapped; the kernel then reads it over the
 *   host link, with no staging copy -- on Grace-Blackwell the NVLink-C2C).
 *   Pageable host memory is refused.
 * Sources are read only; master, m, v and out are updated in place.
 * Errors: ZERO_EINVAL (null, range outside the owned shards, bad mode/dtype,
 *   hp->step < 1, non-finite hyper-parameter, divisor <= 0, pointer of the
 *   wrong kind), ZERO_ERANGE (n_src > ZERO_MAX_SRC), ZERO_EALIGN, ZERO_ECUDA. */
int zero_reduce_scatter_adamw(const zero_layout_t* L,
                              const void* const* src, int32_t n_src, int32_t src_dtype,
                              int64_t src_base, float divisor,
                              int32_t rank_begin, int32_t rank_end,
                              int64_t begin, int64_t end,
                              float* master, float* m, float* v,
                              uint16_t* out_bf16, int32_t out_mode,
                              const zero_adamw_t* hp, void* stream);

/* ---- the fused update with an 8-bit output (ZeRO++) -----------------------
 * Stage 3 with 8-bit weight gathers ("ZeRO Optimizer, in depth", "Offload and
 * ZeRO++": zero_quantized_weights quantises the weight all-gather): the
 * owner's update writes its shard straight in the 8-bit block format, instead
 * of bf16 that zero_quantize_int8 would read back.
 *
 * Computes exactly zero_reduce_scatter_adamw with ZERO_OUT_SHARD followed by
 * zero_quantize_int8 of the bf16 results with block 256: master/m/v are
 * updated as there; q_out (int8, laid out like master: [i - rank_begin*S])
 * receives the codes of bf16_rne(w), and scales_out one fp32 scale per 256
 * elements of that layout ([(i - rank_begin*S) / 256]); no bf16 is written.
 * Requirements: block == 256; S, begin and end multiples of 256 (lay the unit
 * out with align = 256); master, m, v, q_out and the sources 16-byte aligned
 * at begin (there is no element-wise fallback); scales_out 4-byte aligned.
 * Sources as for zero_reduce_scatter_adamw (bf16 gradients or fp32 buffers).
 * Errors: ZERO_EINVAL (as zero_reduce_scatter_adamw, block, a range or shard
 * off the 256-element grid), ZERO_EALIGN, ZERO_ERANGE, ZERO_ECUDA. */
int zero_reduce_scatter_adamw_q8(const zero_layout_t* L, const void* const* src, int32_t n_src,
                                 int32_t src_dtype, int64_t src_base, float divisor,
                                 int32_t rank_begin, int32_t rank_end, int64_t begin, int64_t end,
                                 float* master, float* m, float* v, int8_t* q_out,
                                 float* scales_out, int32_t block, const zero_adamw_t* hp,
                                 void* stream);

/* ---- clipping by the global gradient norm --------------------------------
 * "DeepSpeed ZeRO", "The configuration file" and "ZeRO Optimizer, in depth",
 * "Running it with DeepSpeed": gradient_clipping 1.0 -- the mean gradient is
 * scaled so that its global L2 norm does not exceed max_norm.
 *
 * zero_grad_norm_sq: for every flat i in [begin, end) forms the mean gradient
 *   g_i exactly as zero_reduce_scatter_adamw does (same sources, base, divisor)
 *   and sums g_i^2: each thread in a compensated pair of fp32 values (about 48
 *   significant bits; squares outside that pair's exact range in fp64), then
 *   fp64 across threads and CTAs.  *norm_sq (DEVICE pointer, 8-byte aligned)
 *   receives the sum (accumulate = 0) or has it added (accumulate = 1, for the
 *   second and later buckets of one step).  Nothing is returned to the host.
 *   The summation order is fixed for a given GPU and range, so results repeat
 *   run to run; against a sequential fp64 sum they differ by about 1e-12
 *   relative.
 *   workspace: DEVICE scratch of at least zero_grad_norm_workspace() bytes,
 *   8-byte aligned, owned by the caller; its contents on entry do not matter and
 *   are overwritten (per-CTA partial sums).  Calls that share a workspace must
 *   not overlap on the GPU (use one stream, or one workspace per stream).
 *   [begin, end) inside [0, P); src_base <= begin.
 *   Errors: ZERO_EINVAL, ZERO_ERANGE (workspace too small, n_src too large),
 *   ZERO_EALIGN, ZERO_ECUDA. */
int zero_grad_norm_workspace(int64_t* bytes);
int zero_grad_norm_sq(const zero_layout_t* L, const void* const* src, int32_t n_src,
                      int32_t src_dtype, int64_t src_base, float divisor, int64_t begin,
                      int64_t end, void* workspace, int64_t workspace_bytes, double* norm_sq,
                      int32_t accumulate, void* stream);

/* zero_grad_norm_sq_static: zero_grad_norm_sq without the workspace argument,
 * for callers that cannot allocate device memory -- for example a plugin that
 * is handed only its input and output buffers by a host framework that owns
 * every allocation on the device, or code that must not call cudaMalloc
 * because of the device-wide synchronization it can imply.  The pages have no
 * counterpart: this is an interface convenience of this library.
 * The per-CTA partial sums live in a library-owned device array sized for
 * GPUs of up to 512 SMs: 512 x (2048 / CTA threads) doubles, that is 4096
 * doubles (32 KiB) in the default build of 256 threads per CTA (16384, 128
 * KiB, in a 64-thread build).  It is allocated when the library is loaded and
 * held by every GPU that loads it until the process exits, so the call
 * allocates nothing and calls no allocating routine.  Limits: a device with
 * more than 512 SMs gets ZERO_ERANGE.  The first call on each device looks up
 * that array's device address (cudaGetSymbolAddress, with that device
 * current) and caches it; make the first call on a device before any stream
 * capture begins.  If the cached address is no longer device memory of the
 * current device (its context was destroyed by cudaDeviceReset and created
 * again), the call looks it up again.  Every call shares the one array and overwrites the partials
 * it reads, so no clearing is needed between calls, but calls whose work
 * overlaps on the GPU (different streams, no ordering between them) race on
 * the array: order them, or use zero_grad_norm_sq with one workspace each.
 * Arguments, results and other errors as zero_grad_norm_sq. */
int zero_grad_norm_sq_static(const zero_layout_t* L, const void* const* src, int32_t n_src,
                             int32_t src_dtype, int64_t src_base, float divisor, int64_t begin,
                             int64_t end, double* norm_sq, int32_t accumulate, void* stream);

/* zero_reduce_scatter_adamw_clip: zero_reduce_scatter_adamw with the mean
 * gradient multiplied, before the update, by
 *   coef = min(1, fp32(max_norm / (sqrt(*norm_sq) + 1e-6)))
 * (the quotient in fp64, rounded once to fp32; the multiply in fp32).
 * norm_sq is a DEVICE pointer, normally written by zero_grad_norm_sq over the
 * whole step's gradient before the first update launch; max_norm > 0. */
int zero_reduce_scatter_adamw_clip(const zero_layout_t* L,
                                   const void* const* src, int32_t n_src, int32_t src_dtype,
                                   int64_t src_base, float divisor,
                                   int32_t rank_begin, int32_t rank_end,
                                   int64_t begin, int64_t end,
                                   float* master, float* m, float* v,
                                   uint16_t* out_bf16, int32_t out_mode,
                                   const zero_adamw_t* hp, const double* norm_sq, float max_norm,
                                   void* stream);

/* ---- per-step scalars in device memory ----------------------------------
 * For CUDA-graph replay of steps (and per-step learning-rate schedules): the
 * scalars that change from step to step -- lr and the bias corrections of
 * "ZeRO and FSDP", exercise "A sharded Adam step" -- come from device memory.
 *
 * zero_schedule_fill (host only): table (host, 3 * n_steps floats) receives,
 *   for k = 0..n_steps-1, {lr_k, bc1, bc2} of step t = first_step + k, with
 *   bc1 = 1 - beta1^t and bc2 = 1 - beta2^t computed exactly as for a
 *   by-value step (fp64 from the fp32 betas, rounded once to fp32); lr_k =
 *   lrs[k] (host array of n_steps finite floats), or hp->lr when lrs is NULL.
 *   Errors: ZERO_EINVAL (null, first_step < 1, n_steps < 1, a bad value).
 * zero_schedule_advance (device, one thread, on `stream`): k = *step_index;
 *   sched[0..2] = table[3k .. 3k+2]; *step_index = k + 1.  table (device,
 *   3 * n_steps floats), step_index (device int64, 8-byte aligned) and sched
 *   (device, 3 floats) are the caller's; launching it before a step's updates
 *   (inside the same captured graph) moves them to the next row.  When k is
 *   outside [0, n_steps) nothing is written and zero_status_check reports
 *   ZERO_ERANGE.  Errors: ZERO_EINVAL, ZERO_EALIGN, ZERO_ECUDA. */
int zero_schedule_fill(const zero_adamw_t* hp, int64_t first_step, int64_t n_steps,
                       const float* lrs, float* table);
int zero_schedule_advance(const float* table, int64_t n_steps, int64_t* step_index, float* sched,
                          void* stream);

/* ---- stage-3 gather ------------------------------------------------------
 * "DeepSpeed ZeRO", "Stage 3 step by step" and "ZeRO and FSDP", "FSDP, ZeRO-3
 * inside PyTorch": before a unit (layer) runs, its weights are all-gathered
 * from the n_dp shards into one full buffer, used, then released.
 *
 * full_out[o*S + k] = shards[o][k] for o < unit->n_dp, k < unit->shard; full_out
 * holds unit->padded_n bf16 elements.  shards is a host array of unit->n_dp
 * device pointers, each to unit->shard bf16 elements.  Releasing the gathered
 * buffer is the caller's: it simply reuses the buffer for another unit.
 * Errors: ZERO_EINVAL, ZERO_EALIGN, ZERO_ECUDA. */
int zero_gather_layer(const zero_layout_t* unit, const uint16_t* const* shards,
                      uint16_t* full_out, void* stream);

/* ---- fp32 -> bf16 cast of weights ------------------------------------------
 * "ZeRO and FSDP", "The idea, one stage at a time": the owners cast their
 * updated fp32 master shards to bf16 before the all-gather.  The fused update
 * casts every step; this call casts on its own, for the first bf16 weights of
 * freshly initialised master weights and for bf16 weights rebuilt from
 * restored master weights.
 *
 * dst[i] = bf16 of src[i] for i in [0, n), rounded to nearest, ties to even;
 * values at or beyond the largest finite bf16 plus half an ulp become +-inf,
 * subnormals are kept, and a NaN keeps its sign and top payload bits with the
 * quiet bit set (the upper half of its bits OR 0x0040).  src (n fp32) and dst
 * (n bf16 bit patterns) are DEVICE buffers of the caller, 4- and 2-byte
 * aligned (16-byte alignment of both takes the vector path); they must not
 * overlap.  n = 0 does nothing.
 * Errors: ZERO_EINVAL (n < 0, a null or non-device pointer), ZERO_EALIGN,
 * ZERO_ECUDA. */
int zero_cast_bf16(const float* src, uint16_t* dst, int64_t n, void* stream);

/* ---- stage-3 gather with 8-bit weights (ZeRO++) ---------------------------
 * "ZeRO Optimizer, in depth", "Offload and ZeRO++" (zero_quantized_weights
 * quantises the weight all-gather) and "ZeRO and FSDP", "Fewer bytes on the
 * wire" (the weight all-gather quantized to 8 bits).  Format: each rank's bf16
 * shard in blocks of `block` consecutive elements (block = 256, 512, 1024 or
 * 2048; a shard's last block may be shorter), symmetric int8 with one fp32
 * scale per block: scale = max|w| / 127 (fp32), q = round-half-even(w / scale)
 * clamped to [-127, 127]; an all-zero block has scale 0.  Weights must be finite.
 *
 * zero_quantize_int8: shards_bf16 holds the unit's n_dp shards back to back
 *   (padded_n bf16, rank o's at [o*S]); q receives the same layout in int8 and
 *   scales receives n_dp * ceil(S / block) fp32, rank o's at [o * ceil(S/block)].
 * zero_gather_layer_int8: q_shards[o] (S int8) and scale_shards[o]
 *   (ceil(S / block) fp32) are rank o's quantized shard; full_out (padded_n
 *   bf16) receives full[o*S + k] = bf16_rne(q_o[k] * scale_o[k / block]).
 * Vector kernels need S % 8 == 0, 16-byte aligned bf16 buffers and 8-byte
 * aligned int8 buffers; anything else runs element by element on the GPU.
 * Errors: ZERO_EINVAL (null, bad block, pointer kind), ZERO_EALIGN, ZERO_ECUDA. */
int zero_quantize_int8(const zero_layout_t* unit, const uint16_t* shards_bf16, int8_t* q,
                       float* scales, int32_t block, void* stream);
int zero_gather_layer_int8(const zero_layout_t* unit, const int8_t* const* q_shards,
                           const float* const* scale_shards, int32_t block, uint16_t* full_out,
                           void* stream);

/* ---- reduce-scatter of 8-bit gradients (ZeRO++) ---------------------------
 * "ZeRO Optimizer, in depth", "Offload and ZeRO++" (zero_quantized_gradients
 * quantises the gradient reduce-scatter) and "ZeRO and FSDP", "Fewer bytes on
 * the wire" (gradients quantized during the reduce-scatter).  The pages give
 * no format; the one taken is the 8-bit block format above, applied by each
 * rank to its bf16 gradient slice for every owner: rank r calls
 * zero_quantize_int8 with its whole gradient (padded_n bf16) as the "shards",
 * giving codes q_r (padded_n int8, slice o at [o*S]) and scales s_r
 * (n_dp * nb fp32, nb = ceil(S / block), slice o's at [o*nb]).
 *
 * For flat i in [begin, end), owned by o = i / S, with k = i - o*S:
 *   g_r = fp32(q_r[i]) * s_r[o*nb + k/block]      (one fp32 rounding)
 *   x   = +0 + g_0 + g_1 + ... + g_{n_src-1}      (fp32, ascending r)
 * zero_reduce_scatter_adamw_int8: g = x / divisor, then AdamW, the bf16 cast
 *   and the write exactly as zero_reduce_scatter_adamw (state of i at
 *   [i - rank_begin*S]; out at [i] for ZERO_OUT_FULL, like the state for
 *   ZERO_OUT_SHARD); [begin, end) must lie in the owned range of ranks
 *   rank_begin..rank_end-1.
 * zero_accumulate_int8: dst[i - dst_base] = x (first != 0) or
 *   dst[i - dst_base] + x (first == 0) -- the stage-3 layer reduce-scatter
 *   (first = 1, divisor applied by the update) or stage-2 accumulation.
 * q_src and scale_src are host arrays of n_src device pointers; the codes are
 * read at flat offsets [begin, end), the scales of the owners met.  A call runs
 * on `stream`: one launch when [begin, end) is whole shards and every slice
 * qualifies for the vector kernels, else one launch per owner met, in order.
 * Vector kernels need the slice-local start k a multiple of 8, 8-byte aligned
 * codes at `begin` and 16-byte aligned state, output and dst; anything else
 * runs element by element on the GPU.  Gradients must be finite.
 * Errors: ZERO_EINVAL (null, block not 256/512/1024/2048, range, pointer kind,
 * hyper-parameters), ZERO_ERANGE (n_src > ZERO_MAX_SRC), ZERO_EALIGN (scales
 * not 4-byte aligned, state or dst not element-aligned), ZERO_ECUDA. */
int zero_reduce_scatter_adamw_int8(const zero_layout_t* L, const int8_t* const* q_src,
                                   const float* const* scale_src, int32_t n_src, int32_t block,
                                   float divisor, int32_t rank_begin, int32_t rank_end,
                                   int64_t begin, int64_t end, float* master, float* m, float* v,
                                   uint16_t* out_bf16, int32_t out_mode, const zero_adamw_t* hp,
                                   void* stream);
/* zero_reduce_scatter_adamw_int8_q8: zero_reduce_scatter_adamw_int8 with the
 * 8-bit output of zero_reduce_scatter_adamw_q8 -- the owners' update from
 * 8-bit gradients writes their shards straight in the 8-bit block format
 * (out_block == 256): q_out laid out like master, scales_out one per 256
 * elements of it; no bf16 is written.  Same requirements as
 * zero_reduce_scatter_adamw_q8 (S, begin, end on the 256-element grid,
 * aligned buffers, the vector path only). */
int zero_reduce_scatter_adamw_int8_q8(const zero_layout_t* L, const int8_t* const* q_src,
                                      const float* const* scale_src, int32_t n_src, int32_t block,
                                      float divisor, int32_t rank_begin, int32_t rank_end,
                                      int64_t begin, int64_t end, float* master, float* m, float* v,
                                      int8_t* q_out, float* scales_out, int32_t out_block,
                                      const zero_adamw_t* hp, void* stream);
int zero_accumulate_int8(const zero_layout_t* L, const int8_t* const* q_src,
                         const float* const* scale_src, int32_t n_src, int32_t block, float* dst,
                         int64_t dst_base, int64_t begin, int64_t end, int32_t first, void* stream);

/* ---- gradient accumulation / stage-3 layer reduce-scatter ----------------
 * "ZeRO and FSDP", "The idea, one stage at a time", paragraph on gradient
 * accumulation: stage 1 adds each micro-batch's full local gradient into a full
 * buffer and communicates once per step; stage 2 (and stage 3) must
 * reduce-scatter after every micro-batch.  Also the stage-3 per-layer gradient
 * reduce-scatter ("Stage 3 step by step", step 4).
 *
 * For every flat index i in [begin, end):
 *   ZERO_ACC_LOCAL  (n_src == 1): x = src[0][i - src_base]
 *   ZERO_ACC_REDUCE (n_src >= 1): x = sum over r of src[r][i - src_base]
 *                                  (fp32, ascending r, from +0.0f)
 *   dst[i - dst_base] = first ? x : dst[i - dst_base] + x
 * The result is a sum; the mean's division happens in
 * zero_reduce_scatter_adamw (divisor n_dp*K).  [begin, end) inside [0, P);
 * src_base <= begin; dst_base <= begin.
 * Errors: ZERO_EINVAL, ZERO_ERANGE, ZERO_EALIGN, ZERO_ECUDA. */
int zero_accumulate(const zero_layout_t* L, int32_t mode,
                    const void* const* src, int32_t n_src, int32_t src_dtype, int64_t src_base,
                    float* dst, int64_t dst_base, int64_t begin, int64_t end,
                    int32_t first, void* stream);

/* ---- the last micro-batch of an accumulation window, fused with the update --
 * The same sums as zero_accumulate on the last micro-batch followed by
 * zero_reduce_scatter_adamw over the fp32 buffers, in the same order (so
 * bit-identical to that sequence), without writing and re-reading the fp32
 * buffers.  For every flat i in [begin, end):
 *   ZERO_ACC_LOCAL  (stage 1; n_acc == n_grads == number of ranks):
 *       g = (sum over r of (acc[r][i - acc_base] + grads[r][i - grad_base])) / divisor
 *   ZERO_ACC_REDUCE (stage 2; n_acc == 1):
 *       g = (acc[0][i - acc_base] + sum over r of grads[r][i - grad_base]) / divisor
 * (sums in fp32, ranks ascending from +0.0f), then the AdamW update, cast and
 * output exactly as zero_reduce_scatter_adamw.  acc (fp32) and grads (bf16) are
 * host arrays of device pointers, read only.  divisor is n_dp * K for K
 * micro-batches.  Errors as zero_reduce_scatter_adamw. */
int zero_accumulate_adamw(const zero_layout_t* L, int32_t mode,
                          const float* const* acc, int32_t n_acc, int64_t acc_base,
                          const uint16_t* const* grads, int32_t n_grads, int64_t grad_base,
                          float divisor, int32_t rank_begin, int32_t rank_end,
                          int64_t begin, int64_t end, float* master, float* m, float* v,
                          uint16_t* out_bf16, int32_t out_mode, const zero_adamw_t* hp,
                          void* stream);

/* ---- sharded checkpoints ---------------------------------------------------
 * "ZeRO Optimizer, in depth", "Checkpoints: sharded on the way in, consolidated
 * on the way out": every rank writes its own shard of model and optimizer
 * state plus a small metadata file; a consolidation step rebuilds one plain
 * full-precision state, and a layout change (another GPU count) needs a
 * conversion.  These calls handle one rank's shard file; HOST buffers only
 * (the caller copies device shards to host memory and back).
 *
 * File: a fixed header (magic "ZGBSHARD", version 1, the header struct below,
 * a flag for bf16 weights, the CRC-32 of the payload) followed by master[S],
 * m[S], v[S] (fp32) and, when w_bf16 is given, the rank's bf16 weights[S].
 * zero_ckpt_write_shard: ZERO_EINVAL (inconsistent header), ZERO_EIO.
 * zero_ckpt_read_header: reads and checks magic and version only.
 * zero_ckpt_read_shard: capacity = elements each output holds; checks magic,
 *   version and the payload CRC (ZERO_ECORRUPT), the size (ZERO_ERANGE); w_bf16
 *   may be NULL even when the file holds bf16 weights.
 * zero_crc32: the reflected CRC-32 of IEEE 802.3 (poly 0xEDB88320). */
typedef struct {
    int64_t n;            /* real elements of the flat vector */
    int64_t padded_n;     /* n_dp * shard */
    int64_t shard;        /* S */
    int64_t align;
    int64_t step;         /* optimizer steps taken (t of the last update) */
    int32_t n_dp;
    int32_t rank;         /* whose shard this file holds */
    float lr, beta1, beta2, eps, weight_decay;
    int32_t reserved;
} zero_ckpt_header_t;

int zero_ckpt_write_shard(const char* path, const zero_ckpt_header_t* h, const float* master,
                          const float* m, const float* v, const uint16_t* w_bf16);
int zero_ckpt_read_header(const char* path, zero_ckpt_header_t* h, int32_t* has_bf16);
/* The payload CRC-32 recorded in a shard file's header (the header alone is
 * read; zero_ckpt_read_shard verifies the payload against it).  ZERO_EINVAL
 * (null), ZERO_EIO (cannot open), ZERO_ECORRUPT (bad magic or version). */
int zero_ckpt_payload_crc(const char* path, uint32_t* crc);
int zero_ckpt_read_shard(const char* path, zero_ckpt_header_t* h, float* master, float* m,
                         float* v, uint16_t* w_bf16, int64_t capacity);
uint32_t zero_crc32(const void* data, int64_t n);

/* ---- status ---------------------------------------------------------------
 * Synchronizes `stream` and returns ZERO_ECUDA if it (or an earlier launch on
 * this thread) failed; ZERO_ETIMEOUT if a bounded device-side wait (the
 * mbarrier waits of the TMA-staged update) gave up since the last check -- the
 * kernel that gave up recorded it, drained its own copies and returned, so
 * the context stays usable; the record is cleared by this call.  ZERO_ERANGE
 * if a zero_schedule_advance found its index past the table since the last
 * check (also cleared).  Else ZERO_OK.  The only call that waits on the GPU. */
int zero_status_check(void* stream);

/* Launches one CTA that waits on an mbarrier nothing ever completes, bounded
 * by limit_cycles SM cycles (1 .. 2^32): the wait gives up, records
 * ZERO_ETIMEOUT for zero_status_check and the kernel returns.  For testing the
 * failure path of bounded waits without faulting or hanging the GPU.
 * ZERO_EINVAL for a limit out of range. */
int zero_selftest_bounded_wait(int64_t limit_cycles, void* stream);

/* Static string for a status code (never NULL). */
const char* zero_strerror(int code);

/* The name of the last CUDA error behind a ZERO_ECUDA on this thread
 * ("cudaSuccess" if none), for diagnostics. */
const char* zero_last_cuda_error(void);

/* ---- accounting helpers (host-only) ---------------------------------------
 * "ZeRO and FSDP", "Memory per GPU": model-state bytes per GPU with 2-byte
 * weights and gradients and k_bytes of optimizer state per parameter:
 * stage 0: 16N, 1: 4N + 12N/n_dp, 2: 2N + 14N/n_dp, 3: 16N/n_dp (for k = 12).
 * "ZeRO and FSDP", "Communication volume": bytes each GPU sends per step under
 * ring collectives with the exact (n_dp-1)/n_dp factor.
 * ZERO_EINVAL for a stage outside 0..3, n_dp < 1, n < 0 or null out. */
int zero_memory_bytes(double n, int32_t n_dp, int32_t stage, double k_bytes, double* out);
int zero_comm_bytes(double n, int32_t n_dp, int32_t stage, double param_bytes,
                    double grad_bytes, double* out);

/* The learning rate of optimizer step t (t >= 1) under the "WarmupDecayLR"
 * schedule of the example configuration in "DeepSpeed ZeRO", "The
 * configuration file" (warmup_min_lr, warmup_max_lr, warmup_num_steps,
 * total_num_steps).  The page names the schedule and its four parameters but
 * not its shape; the reading taken: with k = t - 1 schedule steps taken,
 *   k <  warmup:          lr = min + (max - min) * k / warmup   (linear warmup)
 *   warmup <= k < total:  lr = max * (total - k) / (total - warmup)
 *                                                     (linear decay to 0)
 *   k >= total:           lr = 0
 * evaluated in double precision and rounded once to float.  Host only.
 * ZERO_EINVAL for t < 1, warmup < 0, total <= warmup, non-finite or negative
 * rates, or a null out. */
int zero_lr_warmup_decay(int64_t t, double min_lr, double max_lr, int64_t warmup_steps,
                         int64_t total_steps, float* lr_out);

#ifdef __cplusplus
}
#endif

#endif /* ZERO_GB300_H */
