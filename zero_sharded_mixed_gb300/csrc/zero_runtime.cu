// Host-side runtime support shared by the kernels: pointer checks, device
// properties, launch status, and zero_status_check.
#include <atomic>
#include <map>
#include <mutex>
#include <tuple>

#include "zero_update.cuh"

namespace zgb {
// Reads and clears the status word of the opt-in staged 8-bit gradient
// kernel's bounded waits (zero_qgrad.cu): ZERO_OK or ZERO_ETIMEOUT.
int take_qgrad_status();
}  // namespace zgb

namespace zgb {

int check_device_ptr(const void* p) {
    cudaPointerAttributes a;
    const cudaError_t e = cudaPointerGetAttributes(&a, p);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();   // clear the sticky-free error so later launches are not blamed
        return ZERO_EINVAL;
    }
    if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged) return ZERO_EINVAL;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || a.device != dev) return ZERO_EINVAL;
    return ZERO_OK;
}

int check_source_ptr(const void* p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return ZERO_EINVAL;
    }
    if (a.type == cudaMemoryTypeHost)                       // pinned, mapped at the same address
        return a.devicePointer == p ? ZERO_OK : ZERO_EINVAL;
    return check_device_ptr(p);
}

namespace {
constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];
}  // namespace

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 1;
    if (dev >= kMaxDevices) {
        int n = 1;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        return n > 0 ? n : 1;
    }
    int n = g_sm_count[dev].load(std::memory_order_relaxed);
    if (n <= 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 1;
        g_sm_count[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

int ctas_per_sm(const void* kernel, int threads, size_t smem) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return 1;
    }
    static std::mutex mu;
    static std::map<std::tuple<const void*, int, size_t, int>, int> cache;
    const auto key = std::make_tuple(kernel, threads, smem, dev);
    {
        std::lock_guard<std::mutex> lock(mu);
        const auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess || n < 1) {
        (void)cudaGetLastError();
        n = 1;
    }
    std::lock_guard<std::mutex> lock(mu);
    cache[key] = n;
    return n;
}

namespace {
thread_local cudaError_t g_last_error = cudaSuccess;
}  // namespace

int launch_status() {
    const cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) return ZERO_OK;
    g_last_error = e;
    return ZERO_ECUDA;
}

void note_cuda_error(cudaError_t e) {
    if (e != cudaSuccess) g_last_error = e;
}

const char* last_cuda_error_name() {
    return g_last_error == cudaSuccess ? "cudaSuccess" : cudaGetErrorName(g_last_error);
}

}  // namespace zgb

extern "C" const char* zero_last_cuda_error(void) { return zgb::last_cuda_error_name(); }

extern "C" int zero_status_check(void* stream) {
    const cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    const cudaError_t last = cudaGetLastError();
    zgb::note_cuda_error(e);
    zgb::note_cuda_error(last);
    if (e != cudaSuccess || last != cudaSuccess) return ZERO_ECUDA;
    const int rc = zgb::take_device_status();   // ZERO_ETIMEOUT if a bounded device wait gave up
    const int rq = zgb::take_qgrad_status();    // the same for the 8-bit gradient kernels' waits
    const int rs = zgb::take_schedule_status();  // ZERO_ERANGE if a schedule index left its table
    return rc != ZERO_OK ? rc : rq != ZERO_OK ? rq : rs;
}
