/* The C ABI from plain C: no Python, no torch.
 *
 *   abi_smoke          host-only calls (layout, ranges, formulas, strerror,
 *                      argument checks that return before any CUDA call)
 *   abi_smoke --gpu    also the cast of the master weights and two fused
 *                      ZeRO steps on the GPU (cudaMalloc'd buffers, the
 *                      default stream), checked against the oracle linked
 *                      into this test program.
 *
 * Test infrastructure: it links both the library and the oracle; neither of
 * them links the other.  Exit status 0 = pass. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "zero_gb300.h"

/* from the oracle (oracle/zero_oracle.c) */
int oracle_layout(const int64_t* numel, int32_t n_tensors, int32_t n_dp, int64_t align,
                  int64_t bucket, int64_t* offsets, int64_t* out);
int oracle_zero_step(const uint16_t* grads, int32_t n_dp, int64_t shard, float* w, float* m,
                     float* v, uint16_t* full_w, int32_t n_copies, float lr, float b1, float b2,
                     float eps, float wd, int64_t t);
uint16_t oracle_f32_to_bf16(float x);

/* the CUDA runtime calls the GPU part needs (declared here to keep the file plain C) */
int cudaMalloc(void** p, size_t n);
int cudaFree(void* p);
int cudaMemcpy(void* dst, const void* src, size_t n, int kind);   /* 1: H2D, 2: D2H */
int cudaDeviceSynchronize(void);

#define CHECK(cond, ...) do { if (!(cond)) { fprintf(stderr, "FAIL %s:%d: ", __FILE__, __LINE__); \
    fprintf(stderr, __VA_ARGS__); fprintf(stderr, "\n"); return 1; } } while (0)

static uint64_t rng_state = 0x9E3779B97F4A7C15ull;
static double rnd(void) {   /* xorshift64*, uniform in (0, 1) */
    rng_state ^= rng_state >> 12; rng_state ^= rng_state << 25; rng_state ^= rng_state >> 27;
    return ((rng_state * 0x2545F4914F6CDD1Dull) >> 11) * (1.0 / 9007199254740992.0) + 1e-300;
}
static float gauss(void) { return (float)(sqrt(-2.0 * log(rnd())) * cos(6.283185307179586 * rnd())); }

static int host_part(void) {
    const int64_t numel[3] = {1000, 3, 4097};
    int64_t offs[3], ref_offs[3], ref[5];
    zero_layout_t L;
    CHECK(zero_layout(numel, 3, 4, 8, 1000, offs, &L) == ZERO_OK, "zero_layout");
    CHECK(oracle_layout(numel, 3, 4, 8, 1000, ref_offs, ref) == 0, "oracle_layout");
    CHECK(L.n == ref[0] && L.shard == ref[1] && L.padded_n == ref[2] && L.bucket == ref[3] &&
          L.n_buckets == ref[4], "layout differs from the oracle");
    CHECK(memcmp(offs, ref_offs, sizeof offs) == 0, "offsets differ");
    int64_t b0, b1, v;
    CHECK(zero_bucket_range(&L, L.n_buckets - 1, &b0, &b1) == ZERO_OK && b1 == L.padded_n, "bucket");
    CHECK(zero_shard_range(&L, 3, &b0, &b1, &v) == ZERO_OK && v == L.n, "shard range");
    double mem;
    CHECK(zero_memory_bytes(7.5e9, 64, 1, 12, &mem) == ZERO_OK && fabs(mem / 1e9 - 31.40625) < 1e-9,
          "memory formula");
    CHECK(zero_layout(numel, 3, 0, 8, 1000, offs, &L) == ZERO_EINVAL, "n_dp = 0 accepted");
    CHECK(strcmp(zero_strerror(ZERO_EALIGN), "misaligned pointer") == 0, "strerror");
    /* an argument error returns before any CUDA call */
    zero_adamw_t hp = {1e-4f, 0.9f, 0.999f, 1e-8f, 0.1f, 0, 0};   /* step 0: invalid */
    const void* src[1] = {(const void*)0x10000};
    float* f = (float*)0x10000;
    uint16_t* o = (uint16_t*)0x10000;
    CHECK(zero_layout(numel, 3, 4, 8, 1000, offs, &L) == ZERO_OK, "layout");
    CHECK(zero_reduce_scatter_adamw(&L, src, 1, ZERO_BF16, 0, 4.0f, 0, 4, 0, 64, f, f, f, o,
                                    ZERO_OUT_FULL, &hp, NULL) == ZERO_EINVAL, "step 0 accepted");
    CHECK(zero_cast_bf16(NULL, NULL, 16, NULL) == ZERO_EINVAL, "null cast buffers accepted");
    CHECK(zero_cast_bf16(NULL, NULL, -1, NULL) == ZERO_EINVAL, "negative cast length accepted");
    return 0;
}

static int gpu_part(void) {
    const int n_dp = 4;
    const int64_t numel[1] = {200003};
    zero_layout_t L;
    CHECK(zero_layout(numel, 1, n_dp, 8, 50000, NULL, &L) == ZERO_OK, "layout");
    const int64_t P = L.padded_n, S = L.shard, N = L.n;
    uint16_t* g = calloc((size_t)(n_dp * P), 2);
    float* w = calloc((size_t)P, 4); float* m = calloc((size_t)P, 4); float* vv = calloc((size_t)P, 4);
    uint16_t* ref_out = calloc((size_t)P, 2); uint16_t* out = calloc((size_t)P, 2);
    float* w2 = calloc((size_t)P, 4); float* m2 = calloc((size_t)P, 4); float* v2 = calloc((size_t)P, 4);
    for (int64_t i = 0; i < N; ++i) w[i] = 0.02f * gauss();
    for (int r = 0; r < n_dp; ++r)
        for (int64_t i = 0; i < N; ++i) g[r * P + i] = oracle_f32_to_bf16(1e-3f * gauss());
    void *dg, *dw, *dm, *dv, *dout;
    CHECK(cudaMalloc(&dg, (size_t)(n_dp * P * 2)) == 0 && cudaMalloc(&dw, (size_t)P * 4) == 0 &&
          cudaMalloc(&dm, (size_t)P * 4) == 0 && cudaMalloc(&dv, (size_t)P * 4) == 0 &&
          cudaMalloc(&dout, (size_t)P * 2) == 0, "cudaMalloc");
    cudaMemcpy(dg, g, (size_t)(n_dp * P * 2), 1);
    cudaMemcpy(dw, w, (size_t)P * 4, 1); cudaMemcpy(dm, m, (size_t)P * 4, 1); cudaMemcpy(dv, vv, (size_t)P * 4, 1);
    const void* src[4];
    for (int r = 0; r < n_dp; ++r) src[r] = (const char*)dg + (size_t)(r * P * 2);
    memcpy(w2, w, (size_t)P * 4);
    /* the first bf16 weights: the library's cast of the master weights, every
       element equal to the oracle's round-to-nearest-even conversion */
    CHECK(zero_cast_bf16((const float*)dw, (uint16_t*)dout, P, NULL) == ZERO_OK, "zero_cast_bf16");
    CHECK(cudaDeviceSynchronize() == 0, "sync");
    cudaMemcpy(out, dout, (size_t)P * 2, 2);
    for (int64_t i = 0; i < P; ++i)
        CHECK(out[i] == oracle_f32_to_bf16(w[i]), "cast differs from the oracle at %lld", (long long)i);
    for (int64_t t = 1; t <= 2; ++t) {
        zero_adamw_t hp = {1e-4f, 0.9f, 0.999f, 1e-8f, 0.1f, 0, t};
        for (int64_t b = 0; b < L.n_buckets; ++b) {
            int64_t lo, hi;
            CHECK(zero_bucket_range(&L, b, &lo, &hi) == ZERO_OK, "bucket");
            int rc = zero_reduce_scatter_adamw(&L, src, n_dp, ZERO_BF16, 0, (float)n_dp, 0, n_dp, lo, hi,
                                               (float*)dw, (float*)dm, (float*)dv, (uint16_t*)dout,
                                               ZERO_OUT_FULL, &hp, NULL);
            CHECK(rc == ZERO_OK, "zero_reduce_scatter_adamw: %s", zero_strerror(rc));
        }
        CHECK(oracle_zero_step(g, n_dp, S, w2, m2, v2, ref_out, 1, 1e-4f, 0.9f, 0.999f, 1e-8f, 0.1f, t) == 0,
              "oracle");
    }
    CHECK(zero_status_check(NULL) == ZERO_OK, "status");
    cudaMemcpy(w, dw, (size_t)P * 4, 2); cudaMemcpy(m, dm, (size_t)P * 4, 2); cudaMemcpy(vv, dv, (size_t)P * 4, 2);
    cudaMemcpy(out, dout, (size_t)P * 2, 2);
    CHECK(memcmp(w, w2, (size_t)P * 4) == 0 && memcmp(m, m2, (size_t)P * 4) == 0 &&
          memcmp(vv, v2, (size_t)P * 4) == 0, "state differs from the oracle");
    CHECK(memcmp(out, ref_out, (size_t)P * 2) == 0, "bf16 weights differ from the oracle");
    /* a host pointer is refused before any launch */
    zero_adamw_t hp = {1e-4f, 0.9f, 0.999f, 1e-8f, 0.1f, 0, 3};
    CHECK(zero_reduce_scatter_adamw(&L, src, n_dp, ZERO_BF16, 0, 4.0f, 0, n_dp, 0, 64, w, (float*)dm,
                                    (float*)dv, (uint16_t*)dout, ZERO_OUT_FULL, &hp, NULL) == ZERO_EINVAL,
          "host pointer accepted");
    cudaFree(dg); cudaFree(dw); cudaFree(dm); cudaFree(dv); cudaFree(dout);
    free(g); free(w); free(m); free(vv); free(ref_out); free(out); free(w2); free(m2); free(v2);
    return 0;
}

int main(int argc, char** argv) {
    if (host_part()) return 1;
    if (argc > 1 && strcmp(argv[1], "--gpu") == 0 && gpu_part()) return 1;
    printf("abi_smoke ok%s\n", argc > 1 ? " (gpu)" : "");
    return 0;
}
