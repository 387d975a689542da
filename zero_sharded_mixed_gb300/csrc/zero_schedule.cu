// Per-step scalars in device memory, for CUDA-graph replay of steps and for
// per-step learning-rate schedules.
//
// The update kernels read lr and the bias corrections of the step ("ZeRO and
// FSDP", exercise "A sharded Adam step": 1 - beta^t at step t) from
// zero_adamw_t::sched when it is set.  zero_schedule_fill computes a table of
// them on the host, with the same function as the by-value path, so the
// results are bit-identical to it; zero_schedule_advance, one thread, copies
// the current row into sched and moves a device step index on -- launched
// inside a captured graph before the step's updates, it makes every replay
// the next step.
#include <cmath>

#include "zero_update.cuh"

namespace zgb {

__device__ int g_schedule_status;   // ZERO_OK, or ZERO_ERANGE once the index left the table

__global__ void schedule_advance_kernel(const float* table, int64_t n_steps, int64_t* step_index,
                                        float* sched) {
    const int64_t k = *step_index;
    if (k < 0 || k >= n_steps) {
        atomicExch(&g_schedule_status, ZERO_ERANGE);
        return;
    }
    sched[0] = table[3 * k];
    sched[1] = table[3 * k + 1];
    sched[2] = table[3 * k + 2];
    *step_index = k + 1;
}

int take_schedule_status() {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_schedule_status, sizeof v) != cudaSuccess) {
        (void)cudaGetLastError();
        return ZERO_ECUDA;
    }
    if (v != ZERO_OK) {
        const int zero = ZERO_OK;
        if (cudaMemcpyToSymbol(g_schedule_status, &zero, sizeof zero) != cudaSuccess) {
            (void)cudaGetLastError();
            return ZERO_ECUDA;
        }
    }
    return v == ZERO_OK ? ZERO_OK : ZERO_ERANGE;
}

}  // namespace zgb

extern "C" int zero_schedule_fill(const zero_adamw_t* hp, int64_t first_step, int64_t n_steps,
                                  const float* lrs, float* table) {
    if (!hp || !table || first_step < 1 || n_steps < 1) return ZERO_EINVAL;
    if (n_steps > INT64_MAX - first_step || n_steps > INT64_MAX / 3) return ZERO_EINVAL;   // step and index in range
    if (!(hp->beta1 >= 0.0f && hp->beta1 < 1.0f) || !(hp->beta2 >= 0.0f && hp->beta2 < 1.0f))
        return ZERO_EINVAL;
    for (int64_t k = 0; k < n_steps; ++k) {
        const float lr = lrs ? lrs[k] : hp->lr;
        if (!std::isfinite(lr)) return ZERO_EINVAL;
        float bc1 = 0.0f, bc2 = 0.0f;
        zgb::bias_corrections(hp->beta1, hp->beta2, first_step + k, &bc1, &bc2);
        if (!(bc1 > 0.0f) || !(bc2 > 0.0f)) return ZERO_EINVAL;
        table[3 * k] = lr;
        table[3 * k + 1] = bc1;
        table[3 * k + 2] = bc2;
    }
    return ZERO_OK;
}

extern "C" int zero_schedule_advance(const float* table, int64_t n_steps, int64_t* step_index,
                                     float* sched, void* stream) {
    using namespace zgb;
    if (!table || !step_index || !sched || n_steps < 1) return ZERO_EINVAL;
    if (check_aligned(table, 4) || check_aligned(sched, 4) || check_aligned(step_index, 8))
        return ZERO_EALIGN;
    if (check_device_ptr(table) || check_device_ptr(step_index) || check_device_ptr(sched))
        return ZERO_EINVAL;
    schedule_advance_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(table, n_steps, step_index, sched);
    return launch_status();
}
