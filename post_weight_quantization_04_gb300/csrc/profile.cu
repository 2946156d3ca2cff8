// profile.cu — launch counting and optional per-kernel CUDA-event timing.
//
// Every kernel launch in the library goes through GPTQ_LAUNCH (common.cuh), which bumps
// a process-wide counter and, while profiling is enabled, brackets the launch with two
// CUDA events on the launching stream. gptq_profile_read() waits for the recorded events
// and returns per-kernel totals (launches and milliseconds), then clears them.
#include <mutex>
#include <vector>

#include "common.cuh"

namespace gptq {

std::atomic<unsigned long long> g_launches{0};
std::atomic<int> g_profiling{0};

namespace {

struct Rec {
    int id;
    cudaEvent_t a, b;
};

std::mutex g_mu;
std::vector<Rec> g_recs;
std::vector<cudaEvent_t> g_pool;
thread_local cudaEvent_t t_open = nullptr;
thread_local int t_open_id = -1;

cudaEvent_t take_event() {
    if (!g_pool.empty()) {
        cudaEvent_t e = g_pool.back();
        g_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    return e;
}

const char* kNames[K_COUNT] = {
    "hessian_tc_kernel",   "hessian_simt_kernel", "finalize_kernel",   "prep_diag_kernel",
    "prep_perm_kernel",    "prep_gather_kernel",  "potrf_diag_kernel", "sgemm_kernel[prepare]",
    "eye_kernel",          "prep_scatter_kernel", "init_work_kernel",  "row_params_kernel",
    "gptq_block_kernel",   "sgemm_kernel[trailing]", "g_idx_kernel",
    "pack_kernel",         "rtn_kernel",          "split_kernel",      "tc_gemm_nt_kernel[prepare]",
    "tc_gemm_nt_kernel[trailing]", "dequant_matmul_kernel", "merge_status_kernel",
    "tc_gemm_nt_kernel[chain]",
};

}  // namespace

void prof_begin(int id, cudaStream_t s) {
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (!g_profiling.load(std::memory_order_relaxed)) return;
    std::lock_guard<std::mutex> lk(g_mu);
    t_open = take_event();
    t_open_id = id;
    if (t_open) cudaEventRecord(t_open, s);
}

void prof_end(int id, cudaStream_t s) {
    if (!g_profiling.load(std::memory_order_relaxed) || !t_open || t_open_id != id) return;
    std::lock_guard<std::mutex> lk(g_mu);
    cudaEvent_t b = take_event();
    if (b) {
        cudaEventRecord(b, s);
        g_recs.push_back(Rec{id, t_open, b});
    } else {
        g_pool.push_back(t_open);
    }
    t_open = nullptr;
    t_open_id = -1;
}

}  // namespace gptq

using namespace gptq;

extern "C" void gptq_profile_enable(int on) { g_profiling.store(on ? 1 : 0); }

extern "C" unsigned long long gptq_launch_count(void) { return g_launches.load(); }

extern "C" int gptq_profile_read(double* ms, unsigned long long* launches, int n) {
    if (n < 0) return GPTQ_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(g_mu);
    for (int i = 0; i < n && i < K_COUNT; ++i) {
        if (ms) ms[i] = 0.0;
        if (launches) launches[i] = 0;
    }
    int rc = GPTQ_OK;
    for (const Rec& r : g_recs) {
        float t = 0.0f;
        if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess) {
            (void)cudaGetLastError();
            rc = GPTQ_ERR_CUDA;
        }
        if (r.id >= 0 && r.id < n && r.id < K_COUNT) {
            if (ms) ms[r.id] += t;
            if (launches) launches[r.id] += 1;
        }
        g_pool.push_back(r.a);
        g_pool.push_back(r.b);
    }
    g_recs.clear();
    return rc;
}

extern "C" int gptq_profile_kernel_count(void) { return K_COUNT; }

extern "C" const char* gptq_profile_kernel_name(int id) {
    return (id >= 0 && id < K_COUNT) ? kNames[id] : "unknown";
}
