// status.cu — how an entry point reports device-side errors (a timed-out wait, a failed
// factorisation, a non-finite input): at once, by synchronising its stream (the default),
// or deferred.
//
// In deferred mode an entry point returns as soon as its work is enqueued; a one-thread
// kernel at the end of its work folds the call's status word into one sticky status word
// per device (first error kept), and gptq_status_sync reads and clears it. A caller that
// enqueues a whole model's calls then pays for one host synchronisation instead of one per
// call, and the GPU does not idle while the host returns and issues the next call.
#include <cuda.h>

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

// per-call status words for the entry points without a workspace (a ring in static device
// memory; see call_status_word)
constexpr int kStatusWords = 256;
__device__ int g_call_status[kStatusWords];
std::atomic<unsigned> g_next_word{0};
ContextPtrCache g_call_status_addr;

using PfnCtxGetCurrent = CUresult (*)(CUcontext*);
using PfnCtxGetId = CUresult (*)(CUcontext, unsigned long long*);

}  // namespace

unsigned long long current_context_id() {
    static PfnCtxGetCurrent get_current = nullptr;
    static PfnCtxGetId get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PfnCtxGetCurrent>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PfnCtxGetId>(f);
        (void)cudaGetLastError();
    });
    if (!get_current || !get_id) return 0;
    CUcontext c = nullptr;
    if (get_current(&c) != CUDA_SUCCESS || !c) return 0;
    unsigned long long id = 0;
    if (get_id(c, &id) != CUDA_SUCCESS) return 0;
    return id + 1;   // 0 stays "no context"
}

cudaError_t call_status_word(cudaStream_t s, int** out) {
    void* base = g_call_status_addr.find(current_context_id());
    if (!base) {
        const cudaError_t e = cudaGetSymbolAddress(&base, g_call_status);
        if (e != cudaSuccess) return e;
        g_call_status_addr.put(current_context_id(), base);   // the lookup made the context current
    }
    int* w = static_cast<int*>(base) + (g_next_word.fetch_add(1, std::memory_order_relaxed) % kStatusWords);
    *out = w;
    return cudaMemsetAsync(w, 0, sizeof(int), s);
}

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
    GPTQ_CUDA_TRY(cudaMemcpyFromSymbolAsync(&hs, g_sticky_status, sizeof(int), 0, cudaMemcpyDeviceToHost, s));
    GPTQ_CUDA_TRY(cudaStreamSynchronize(s));
    if (hs != 0) {
        const int zero = 0;
        GPTQ_CUDA_TRY(cudaMemcpyToSymbol(g_sticky_status, &zero, sizeof(int)));
    }
    return hs;
}

// Test hook, deliberately not declared in gptq.h: sets the limit of every pipeline mbarrier
// wait in the library's kernels (a limit of 0 gives up at the first wait that is not
// already complete, which makes a call report GPTQ_ERR_TIMEOUT and exercises the unwind
// path: in-flight copies and MMAs drained with the full limit, TMEM freed). Not for
// production use. Synchronous (device-wide). Errors: CUDA.
extern "C" int gptq_test_set_wait_limit_ns(unsigned long long ns) {
    GPTQ_CUDA_TRY(cudaDeviceSynchronize());
    GPTQ_CUDA_TRY(hessian_set_wait_limit(ns));
    GPTQ_CUDA_TRY(tc_gemm_set_wait_limit(ns));
    GPTQ_CUDA_TRY(dequant_set_wait_limit(ns));
    return GPTQ_OK;
}
