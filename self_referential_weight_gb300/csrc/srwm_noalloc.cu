// srwm_noalloc.cu -- srwm_forward_balanced for callers that cannot allocate
// device memory.
//
// The balanced schedule needs a small scratch area: one progress counter per
// (sequence, head) stream.  srwm_forward_balanced takes it from the caller.
// Some callers cannot provide it: code that runs under a host framework which
// owns every device allocation and exposes no allocator to plugins, or paths
// that must not call cudaMalloc because of its implicit synchronisation and
// its failure modes at run time.  For them this file keeps the counters in a
// fixed array in the library's own device memory, so the call allocates
// nothing.
//
// The array lives for as long as the library is loaded, on every GPU that
// loads it (kMaxStreams * 4 bytes = 256 KiB each).  In host code the array's
// name only stands for the symbol; its device address is looked up once per
// device with cudaGetSymbolAddress while that device is current.
#include <cuda_runtime.h>

#include <mutex>

#include "srwm.h"

namespace {

// Largest B * H this entry point accepts.
constexpr int kMaxStreams = 65536;

static __device__ __align__(256) int g_noalloc_counters[kMaxStreams];

constexpr int kMaxDevices = 64;
int* g_counter_ptr[kMaxDevices];
std::mutex g_counter_mu;

// Device address of the counter array on the current device.  The first call
// on a device performs the lookup.
int counter_ptr(int** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return SRWM_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lk(g_counter_mu);
    if (!g_counter_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_counters) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return SRWM_ERR_CUDA;
        }
        g_counter_ptr[dev] = static_cast<int*>(p);
    }
    *out = g_counter_ptr[dev];
    return SRWM_OK;
}

}  // namespace

extern "C" int srwm_forward_balanced_noalloc(const float* x, const float* W0, int B, int T, int H, int d,
                                             int n_lr, int softmax_input, float* y_out, float* W_final,
                                             void* stream)
{
    if (B > 0 && H > 0 && static_cast<long long>(B) * H > kMaxStreams) return SRWM_ERR_SHAPE;
    int* counters = nullptr;
    const int rc = counter_ptr(&counters);
    if (rc != SRWM_OK) return rc;
    // srwm_forward_balanced zeroes the counters it uses on `stream` before the
    // kernel runs, so whatever the previous call left there does not matter.
    return srwm_forward_balanced(x, W0, B, T, H, d, n_lr, softmax_input, y_out, W_final, counters,
                                 sizeof(int) * static_cast<size_t>(kMaxStreams), stream);
}
