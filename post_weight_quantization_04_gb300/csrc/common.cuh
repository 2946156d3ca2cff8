// common.cuh — shared helpers for libgptq's sm_103a kernels: status plumbing, bounded
// mbarrier waits, TMA loads and tcgen05 (TMEM / UMMA) wrappers written as inline PTX.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "gptq.h"

#define GPTQ_CUDA_TRY(expr)                                   \
    do {                                                      \
        cudaError_t e_ = (expr);                              \
        if (e_ != cudaSuccess) {                              \
            (void)cudaGetLastError();                         \
            return GPTQ_ERR_CUDA;                             \
        }                                                     \
    } while (0)

#define GPTQ_LAUNCH_CHECK()                                   \
    do {                                                      \
        cudaError_t e_ = cudaGetLastError();                  \
        if (e_ != cudaSuccess) return GPTQ_ERR_CUDA;          \
    } while (0)

namespace gptq {

// Kernel classes for launch counting and per-kernel event timing (profile.cu).
enum KernelId {
    K_HESS_TC, K_HESS_SIMT, K_FINALIZE, K_PREP_DIAG, K_PREP_PERM, K_PREP_GATHER, K_POTRF, K_SGEMM_PREP,
    K_EYE, K_SCATTER, K_INIT_WORK, K_ROW_PARAMS, K_BLOCK, K_SGEMM_TRAIL, K_G_IDX, K_PACK, K_RTN,
    K_SPLIT, K_TC_PREP, K_TC_TRAIL, K_DEQUANT_MM, K_STATUS, K_TC_CHAIN, K_COUNT
};
void prof_begin(int id, cudaStream_t s);
void prof_end(int id, cudaStream_t s);

// Launch through this so every kernel is counted (and timed while profiling is on).
#define GPTQ_LAUNCH(id, stream, ...)            \
    do {                                        \
        ::gptq::prof_begin((id), (stream));     \
        __VA_ARGS__;                            \
        ::gptq::prof_end((id), (stream));       \
    } while (0)

constexpr int kSMs = 152;  // fallback only; the real count is queried per device

int device_sm_count();

// The end of an entry point: report the call's device status word at once (synchronising
// the stream) or, in deferred mode, fold it into the device's sticky status and return OK.
int finish_call(const int* status, cudaStream_t s);

// The unique id of the CUDA context current on this thread (cuCtxGetId: never reused in
// the life of the process, so an address cached under it cannot outlive a device reset or
// belong to another context); 0 when no context is current or the driver lacks the call.
unsigned long long current_context_id();

// A device pointer per CUDA context (the address of a file-scope __device__ array in that
// context), looked up once per context by its owner and kept for the life of the process.
struct ContextPtrCache {
    static constexpr int kEntries = 16;
    std::mutex mu;
    unsigned long long id[kEntries] = {};
    void* ptr[kEntries] = {};
    int n = 0;
    void* find(unsigned long long cid) {
        if (!cid) return nullptr;
        std::lock_guard<std::mutex> lk(mu);
        for (int i = 0; i < n && i < kEntries; ++i)
            if (id[i] == cid) return ptr[i];
        return nullptr;
    }
    void put(unsigned long long cid, void* p) {
        if (!cid) return;
        std::lock_guard<std::mutex> lk(mu);
        const int i = n % kEntries;   // the oldest entry goes first once all are used
        id[i] = cid;
        ptr[i] = p;
        ++n;
    }
};

// A device status word for one call of an entry point that has no workspace (the consumer
// of the stored form, round-to-nearest): one of a ring of words in static device memory
// (nothing is allocated), cleared on `s`. Calls in flight at the same time get different
// words unless a few hundred calls are issued while one is still running.
cudaError_t call_status_word(cudaStream_t s, int** out);

// Test hook support: sets this library's limit on pipeline mbarrier waits (mbar_wait) in
// every translation unit that has such waits; the drain waits keep kWaitLimitNs.
cudaError_t hessian_set_wait_limit(unsigned long long ns);
cudaError_t tc_gemm_set_wait_limit(unsigned long long ns);
cudaError_t dequant_set_wait_limit(unsigned long long ns);

static inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// ------------------------------------------------------------------------------------
// Programmatic dependent launch. A kernel launched with launch_pdl may start while the
// kernel before it in the stream is still running; it must call pdl_wait() before it
// touches any global memory that an earlier kernel writes or reads (everything before
// that point is prologue: shared memory set-up, TMEM allocation, descriptor prefetch,
// loads of data no earlier kernel of the call writes). pdl_trigger() lets the next
// kernel begin its own prologue. In a kernel launched without the attribute both are
// no-ops.
// ------------------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// ------------------------------------------------------------------------------------
// device-side status: kernels record failures into a device int (first error wins)
// ------------------------------------------------------------------------------------
__device__ __forceinline__ void set_status(int* status, int code) {
    if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Every spin-wait in this library gives up after this long, records GPTQ_ERR_TIMEOUT and
// lets the kernel unwind (no kernel waits on another launch or another device).
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// The limit of the pipeline waits (mbar_wait) of this translation unit, kWaitLimitNs unless a
// test lowers it through the library's test hook (a limit of 0 gives up at the first wait
// that is not already complete). The drain waits, which let in-flight copies and MMAs land
// before a CTA exits, always use kWaitLimitNs.
static __device__ unsigned long long g_pipeline_wait_limit_ns = kWaitLimitNs;

static inline cudaError_t set_pipeline_wait_limit_this_unit(unsigned long long ns) {
    return cudaMemcpyToSymbol(g_pipeline_wait_limit_ns, &ns, sizeof(ns));
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------------------------
// mbarrier
// ------------------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with `parity` to complete. Returns false (after recording
// GPTQ_ERR_TIMEOUT and raising the CTA's abort flag) if the limit passes or another
// thread of the CTA already aborted.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int* status) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    const uint64_t limit = *static_cast<volatile unsigned long long*>(&g_pipeline_wait_limit_ns);
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0 || limit == 0) {
            if (*abort_flag) return false;
            if (globaltimer_ns() - t0 >= limit) {
                *abort_flag = 1;
                set_status(status, GPTQ_ERR_TIMEOUT);
                return false;
            }
        }
    }
}

// The same wait for a whole warp with one lane polling: the other 31 lanes do not poll the
// barrier word; once lane 0 has seen the phase complete, each lane's own try_wait succeeds
// at once and gives it the barrier's acquire ordering. Call from all 32 lanes, and only for
// a barrier whose next phase cannot complete before this warp itself arrives somewhere.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                               int* status) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort_flag, status);
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    if (ok) ok = mbar_try_wait(bar, parity);
    return ok;
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------------------------
// TMA (tiled tensor copies global -> shared, completion counted on an mbarrier)
// ------------------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, uint32_t bar, int32_t x,
                                            int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// ------------------------------------------------------------------------------------
// tcgen05: tensor memory allocation, MMA issue/commit, TMEM -> register loads
// ------------------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc], kind::f16 (bf16 inputs here), fp32 accumulate.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every tcgen05.mma this thread issued before has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread t gets lane (base + t), columns c..c+31.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
          "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
          "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

// The store direction: thread t writes lane (base + t), columns c..c+31.
__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor for tcgen05.mma (sm_100 family layout):
//   [0,14) start >> 4 | [16,30) leading byte offset >> 4 | [32,46) stride byte offset >> 4
//   [46,48) version = 1 | [49,52) base offset = 0 | [52] lbo mode = 0 | [61,64) swizzle
// For an MN-major operand in the 128-byte swizzle layout: LBO = byte distance between
// 64-element (128 B) slabs along M/N, SBO = byte distance between 8-row groups along K.
constexpr uint64_t kSwizzle128B = 2;

__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint64_t swz) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (swz & 7ull) << 61;
    return d;
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, both MN-major.
//   [4,6) D fmt (1 = f32) | [7,10) A fmt (1 = bf16) | [10,13) B fmt (1 = bf16)
//   [15] A major (1 = MN) | [16] B major (1 = MN) | [17,23) N >> 3 | [24,29) M >> 4
__host__ __device__ constexpr uint32_t idesc_bf16_f32_mn_mn(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) | (1u << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ------------------------------------------------------------------------------------
// small helpers
// ------------------------------------------------------------------------------------
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_min(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

}  // namespace gptq
