// status.cu — how an entry point reports device-side errors (a timed-out wait, a failed
// factorisation): at once, by synchronising its stream (the default), or deferred.
//
// In deferred mode an entry point returns as soon as its work is enqueued; a one-thread
// kernel at the end of its work folds the call's status word into one sticky status word
// per device (first error kept), and gptq_status_sync reads and clears it. A caller that
// enqueues a whole model's calls then pays for one host synchronisation instead of one per
// call, and the GPU does not idle while the host returns and issues the next call.
#include <atomic>
#include <mutex>

#include "common.cuh"

namespace gptq {

namespace {

std::atomic<int> g_mode{GPTQ_STATUS_SYNC};

// the device's sticky status: static device memory, so no call allocates for it
__device__ int g_sticky_status;

__global__ void merge_status_kernel(const int* __restrict__ status) {
    const int v = *status;
    if (v != 0) atomicCAS(&g_sticky_status, 0, v);
}

}  // namespace

int finish_call(const int* status, cudaStream_t s) {
    if (g_mode.load(std::memory_order_relaxed) == GPTQ_STATUS_DEFERRED) {
        GPTQ_LAUNCH(K_STATUS, s, merge_status_kernel<<<1, 1, 0, s>>>(status));
        GPTQ_LAUNCH_CHECK();
        return GPTQ_OK;
    }
    int hs = 0;
    GPTQ_CUDA_TRY(cudaMemcpyAsync(&hs, status, sizeof(int), cudaMemcpyDeviceToHost, s));
    GPTQ_CUDA_TRY(cudaStreamSynchronize(s));
    return hs;
}

}  // namespace gptq

using namespace gptq;

extern "C" int gptq_set_status_mode(int mode) {
    if (mode != GPTQ_STATUS_SYNC && mode != GPTQ_STATUS_DEFERRED) return GPTQ_ERR_INVALID_ARG;
    g_mode.store(mode);
    return GPTQ_OK;
}

extern "C" int gptq_status_mode(void) { return g_mode.load(); }

extern "C" int gptq_status_sync(void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int hs = 0;
    const int zero = 0;
    GPTQ_CUDA_TRY(cudaMemcpyFromSymbolAsync(&hs, g_sticky_status, sizeof(int), 0, cudaMemcpyDeviceToHost, s));
    GPTQ_CUDA_TRY(cudaMemcpyToSymbolAsync(g_sticky_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s));
    GPTQ_CUDA_TRY(cudaStreamSynchronize(s));
    return hs;
}
