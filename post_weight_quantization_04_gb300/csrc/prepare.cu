// prepare.cu — gptq_prepare: dead inputs, damping, act_order permutation and
// U = upper Cholesky factor of H^-1.
//
// The GPTQ guide page ("Source code", `_hessian_inverse_chol`) forms U as
// cholesky(inv(H)).T. Here the same U comes from one factorisation and one triangular
// inverse, both blocked and fp32 on the GPU:
//
//   Hp  = H[perm][:, perm] with the dead diagonal set to 1 and damping added
//   D   = diag(Hp),   Hh = D^-1/2 Hp D^-1/2            (unit diagonal: equilibration)
//   J   = the reversal permutation,  A = J Hh J = L L^T (ordinary lower Cholesky)
//   then Hh = (J L J)(J L J)^T with J L J upper, so Hh^-1 = Uh^T Uh for Uh = J L^-1 J
//   and U = Uh D^-1/2  satisfies U^T U = Hp^-1 with U upper and a positive diagonal.
//
// Equilibration removes the lognormal per-channel spread of the activations from the
// fp32 factorisation; damping (0.01 * mean diag) bounds the condition number.
//
// Workspace layout (256-byte aligned slabs):
//   A     d*d fp32   reversed, equilibrated Hp -> L (lower triangle)
//   Binv  d*d fp32   identity -> L^-1 (lower triangle)
//   LinvD nblk*NB*NB fp32  inverses of L's diagonal blocks
//   ddiag d fp32, rr d fp32 (1/sqrt(ddiag)), status int
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "sgemm.cuh"
#include "tc_gemm.cuh"

namespace gptq {

namespace {

constexpr int NB = 128;  // panel width of the blocked factorisation

struct PrepWs {
    float* A;
    float* Binv;
    float* LinvD;
    float* ahi;   // d x NB: TF32 split of the GEMM's first operand
    float* alo;
    float* bhi;   // d x NB: TF32 split of the second operand
    float* blo;
    float* ddiag;
    float* rr;
    int* status;
    size_t bytes;
};

constexpr size_t align256c(size_t x) { return (x + 255) & ~size_t(255); }

// slab sizes, in carve order; the total is also the size of the allocation-free scratch
constexpr size_t prep_slab(int64_t d, int i) {
    return i < 2 ? sizeof(float) * d * d
         : i == 2 ? sizeof(float) * ((d + NB - 1) / NB) * NB * NB
         : i < 7 ? sizeof(float) * d * NB
         : i < 9 ? sizeof(float) * d
         : sizeof(int) * 4;
}
constexpr int kPrepSlabs = 10;
constexpr size_t prep_ws_bytes(int64_t d) {
    size_t off = 0;
    for (int i = 0; i < kPrepSlabs; ++i) off = align256c(off + prep_slab(d, i));
    return off;
}

PrepWs carve(void* base, int64_t d) {
    PrepWs w{};
    char* p = static_cast<char*>(base);
    size_t off[kPrepSlabs + 1] = {0};
    for (int i = 0; i < kPrepSlabs; ++i) off[i + 1] = align256c(off[i] + prep_slab(d, i));
    w.A = reinterpret_cast<float*>(p + off[0]);
    w.Binv = reinterpret_cast<float*>(p + off[1]);
    w.LinvD = reinterpret_cast<float*>(p + off[2]);
    w.ahi = reinterpret_cast<float*>(p + off[3]);
    w.alo = reinterpret_cast<float*>(p + off[4]);
    w.bhi = reinterpret_cast<float*>(p + off[5]);
    w.blo = reinterpret_cast<float*>(p + off[6]);
    w.ddiag = reinterpret_cast<float*>(p + off[7]);
    w.rr = reinterpret_cast<float*>(p + off[8]);
    w.status = reinterpret_cast<int*>(p + off[9]);
    w.bytes = off[kPrepSlabs];
    return w;
}

// dead[j] = (H[j][j] == 0); the dead diagonal becomes 1; mean of the fixed diagonal in
// fp64; damped diagonal and its inverse square root.
__global__ void __launch_bounds__(1024) prep_diag_kernel(const float* __restrict__ H, int64_t d, float damp,
                                                        uint8_t* __restrict__ dead, float* __restrict__ ddiag,
                                                        float* __restrict__ rr) {
    __shared__ double part[32];
    double s = 0.0;
    for (int64_t j = threadIdx.x; j < d; j += blockDim.x) {
        const float h = H[j * d + j];
        const bool dj = (h == 0.0f);
        dead[j] = dj ? 1 : 0;
        s += dj ? 1.0 : (double)h;
    }
    s = warp_sum_d(s);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x < 32) {
        double v = (threadIdx.x < (blockDim.x >> 5)) ? part[threadIdx.x] : 0.0;
        v = warp_sum_d(v);
        if (threadIdx.x == 0) part[0] = v;
    }
    __syncthreads();
    const double add = (double)damp * (part[0] / (double)d);
    for (int64_t j = threadIdx.x; j < d; j += blockDim.x) {
        const float h = H[j * d + j];
        const double hd = (h == 0.0f ? 1.0 : (double)h) + add;
        ddiag[j] = (float)hd;
        rr[j] = (float)(1.0 / sqrt(hd));
    }
}

// Stable descending order of the keys: rank(i) = #{k : key_k > key_i} + #{k < i : key_k == key_i};
// perm[rank(i)] = i.
__global__ void __launch_bounds__(256) prep_perm_kernel(const float* __restrict__ key, int64_t d,
                                                       int32_t* __restrict__ perm) {
    __shared__ float tile[256];
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const float ki = (i < d) ? key[i] : 0.0f;
    int64_t rank = 0;
    for (int64_t t0 = 0; t0 < d; t0 += 256) {
        const int64_t k = t0 + threadIdx.x;
        tile[threadIdx.x] = (k < d) ? key[k] : 0.0f;
        __syncthreads();
        const int lim = (int)(d - t0 < 256 ? d - t0 : 256);
        for (int u = 0; u < lim; ++u) {
            const float kk = tile[u];
            rank += (kk > ki) || (kk == ki && t0 + u < i);
        }
        __syncthreads();
    }
    if (i < d) perm[rank] = (int32_t)i;
}

__global__ void iota_kernel(int32_t* __restrict__ perm, int64_t d) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < d) perm[i] = (int32_t)i;
}

// A[i][j] (j <= i) = Hh[d-1-i][d-1-j], Hh = D^-1/2 Hp D^-1/2, Hp = H[perm][:, perm]
// (fixed, damped diagonal; H read from its upper triangle).
__global__ void __launch_bounds__(256) prep_gather_kernel(const float* __restrict__ H, int64_t d,
                                                         const int32_t* __restrict__ perm,
                                                         const float* __restrict__ rr, float* __restrict__ A) {
    const int64_t i = (int64_t)blockIdx.y * 8 + (threadIdx.x >> 5);
    const int64_t jb = (int64_t)blockIdx.x * 32;
    if (i >= d || jb > i) return;
    const int64_t j = jb + (threadIdx.x & 31);
    if (j > i) return;
    const int32_t a = perm[d - 1 - i];
    const int32_t b = perm[d - 1 - j];
    float v;
    if (a == b) {
        v = 1.0f;
    } else {
        const int32_t lo = a < b ? a : b, hi = a < b ? b : a;
        v = H[(int64_t)lo * d + hi] * rr[a] * rr[b];
    }
    A[i * d + j] = v;
}

// One CTA factors the diagonal block A[k0:k0+n, k0:k0+n] = L L^T in place (lower), and
// writes L^-1 (lower, NB x NB, zeros above) to Linv. A non-positive or non-finite pivot
// records GPTQ_ERR_NOT_SPD (and is replaced by 1 so the kernel finishes).
//
// One loop over k produces column k of L (right-looking Cholesky) and applies the matching
// Gauss-Jordan step to X = [I -> L^-1]: X[i][:] -= L[i][k] * X[k][:] / L[k][k] for i > k and
// X[k][:] /= L[k][k]. Everything a thread updates lives in its registers: thread (j, q)
// holds rows 32q..32q+31 of column j of the block, and columns 32q..32q+31 of row j of X.
// At step k the four threads of column k publish the (raw) pivot column, and of row k of X,
// to double-buffered shared arrays; after one barrier every thread updates its registers
// with broadcast reads. Entries above the diagonal of the block are updated too (unused),
// so the update needs no per-element predicate; columns of X beyond k read zeros.
__global__ void __launch_bounds__(512) potrf_diag_kernel(float* __restrict__ A, int64_t lda, int64_t k0, int n,
                                                        float* __restrict__ Linv, int* __restrict__ status) {
    __shared__ __align__(16) float colraw[2][NB];
    __shared__ __align__(16) float xraw[2][NB];
    __shared__ float dg[NB];
    const int tid = threadIdx.x;
    const int q = tid >> 7;                                 // row / column slab 32q..32q+31
    const int j = ((tid & 31) << 2) | ((tid >> 5) & 3);     // column of L, row of X (spread over SMSPs)
    const int r0 = 32 * q;

    float sc[32], xr[32];
#pragma unroll
    for (int t = 0; t < 32; ++t) {
        const int i = r0 + t;
        sc[t] = (i < n && j < n && i >= j) ? A[(k0 + i) * lda + k0 + j] : 0.0f;
        xr[t] = (i == j && j < n) ? 1.0f : 0.0f;
    }

    for (int k = 0; k < n; ++k) {
        const int b = k & 1;
        if (j == k) {
#pragma unroll
            for (int t = 0; t < 32; t += 4) {
                *reinterpret_cast<float4*>(&colraw[b][r0 + t]) = make_float4(sc[t], sc[t + 1], sc[t + 2], sc[t + 3]);
                *reinterpret_cast<float4*>(&xraw[b][r0 + t]) = make_float4(xr[t], xr[t + 1], xr[t + 2], xr[t + 3]);
            }
        }
        __syncthreads();
        float piv = colraw[b][k];
        if (!(piv > 0.0f) || !isfinite(piv)) {
            if (tid == 0) set_status(status, GPTQ_ERR_NOT_SPD);
            piv = 1.0f;
        }
        const float lkk = sqrtf(piv);
        const float inv = 1.0f / lkk;
        if (j > k && j < n) {
            const float f = colraw[b][j] * (inv * inv);     // L[j][k] / L[k][k]
#pragma unroll
            for (int t = 0; t < 32; t += 4) {
                const float4 c4 = *reinterpret_cast<const float4*>(&colraw[b][r0 + t]);
                const float4 x4 = *reinterpret_cast<const float4*>(&xraw[b][r0 + t]);
                sc[t] = fmaf(-c4.x, f, sc[t]);
                sc[t + 1] = fmaf(-c4.y, f, sc[t + 1]);
                sc[t + 2] = fmaf(-c4.z, f, sc[t + 2]);
                sc[t + 3] = fmaf(-c4.w, f, sc[t + 3]);
                xr[t] = fmaf(-f, x4.x, xr[t]);
                xr[t + 1] = fmaf(-f, x4.y, xr[t + 1]);
                xr[t + 2] = fmaf(-f, x4.z, xr[t + 2]);
                xr[t + 3] = fmaf(-f, x4.w, xr[t + 3]);
            }
        } else if (j == k) {
#pragma unroll
            for (int t = 0; t < 32; ++t) {
                sc[t] *= inv;
                xr[t] *= inv;
            }
            if (q == 0) dg[k] = lkk;
        }
    }
    __syncthreads();
#pragma unroll
    for (int t = 0; t < 32; ++t) {
        const int i = r0 + t;
        if (i < n && j < n && i >= j) A[(k0 + i) * lda + k0 + j] = (i == j) ? dg[j] : sc[t];
    }
#pragma unroll
    for (int t = 0; t < 32; t += 4) {
        float4 v;
        v.x = (j < n && r0 + t <= j) ? xr[t] : 0.0f;
        v.y = (j < n && r0 + t + 1 <= j) ? xr[t + 1] : 0.0f;
        v.z = (j < n && r0 + t + 2 <= j) ? xr[t + 2] : 0.0f;
        v.w = (j < n && r0 + t + 3 <= j) ? xr[t + 3] : 0.0f;
        *reinterpret_cast<float4*>(&Linv[j * NB + r0 + t]) = v;
    }
}

__global__ void eye_kernel(float* __restrict__ B, int64_t d) {
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx < d * d) B[idx] = (idx / d == idx % d) ? 1.0f : 0.0f;
}

// U[i][j] = (i <= j) ? Linv[d-1-i][d-1-j] * rr[perm[j]] : 0
__global__ void __launch_bounds__(256) prep_scatter_kernel(const float* __restrict__ Binv, int64_t d,
                                                          const int32_t* __restrict__ perm,
                                                          const float* __restrict__ rr, float* __restrict__ U) {
    const int64_t i = blockIdx.y;
    for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < d; j += (int64_t)gridDim.x * blockDim.x) {
        U[i * d + j] = (i <= j) ? Binv[(d - 1 - i) * d + (d - 1 - j)] * rr[perm[j]] : 0.0f;
    }
}

}  // namespace

}  // namespace gptq

using namespace gptq;

extern "C" size_t gptq_prepare_workspace_bytes(int64_t d, int act_order) {
    (void)act_order;
    if (d <= 0) return 0;
    return carve(nullptr, d).bytes;
}

extern "C" int gptq_prepare(const float* H, const float* diag_xtx, int64_t d, float damp, int act_order, float* U,
                            int32_t* perm, uint8_t* dead, void* ws, size_t ws_bytes, void* stream_) {
    if (d <= 0 || d > (1 << 20) || !H || !U || !perm || !dead || !ws) return GPTQ_ERR_INVALID_ARG;
    if (act_order && !diag_xtx) return GPTQ_ERR_INVALID_ARG;
    if (!(damp >= 0.0f) || !isfinite(damp)) return GPTQ_ERR_INVALID_ARG;
    PrepWs w = carve(ws, d);
    if (ws_bytes < w.bytes) return GPTQ_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream_);

    GPTQ_CUDA_TRY(cudaMemsetAsync(w.status, 0, sizeof(int), s));
    GPTQ_LAUNCH(K_PREP_DIAG, s, prep_diag_kernel<<<1, 1024, 0, s>>>(H, d, damp, dead, w.ddiag, w.rr));
    GPTQ_LAUNCH_CHECK();
    const unsigned g1 = (unsigned)ceil_div(d, 256);
    if (act_order)
        GPTQ_LAUNCH(K_PREP_PERM, s, prep_perm_kernel<<<g1, 256, 0, s>>>(diag_xtx, d, perm));
    else
        GPTQ_LAUNCH(K_PREP_PERM, s, iota_kernel<<<g1, 256, 0, s>>>(perm, d));
    GPTQ_LAUNCH_CHECK();
    {
        dim3 grid((unsigned)ceil_div(d, 32), (unsigned)ceil_div(d, 8));
        GPTQ_LAUNCH(K_PREP_GATHER, s, prep_gather_kernel<<<grid, 256, 0, s>>>(H, d, perm, w.rr, w.A));
        GPTQ_LAUNCH_CHECK();
    }

    const size_t potrf_smem = 0;

    // The trailing contractions run on the tensor cores (3xTF32, operands split into
    // TF32 hi/lo first) when every matrix row is 16-byte aligned, else on the FFMA GEMM.
    const bool tc = (d % 4 == 0) && tc_gemm_nt_ok(w.A, d);

    // blocked right-looking Cholesky of A (lower)
    const int64_t nblk = ceil_div(d, NB);
    for (int64_t kb = 0; kb < nblk; ++kb) {
        const int64_t k0 = kb * NB;
        const int n = (int)std::min<int64_t>(NB, d - k0);
        float* LinvK = w.LinvD + kb * NB * NB;
        GPTQ_LAUNCH(K_POTRF, s, potrf_diag_kernel<<<1, 512, potrf_smem, s>>>(w.A, d, k0, n, LinvK, w.status));
        GPTQ_LAUNCH_CHECK();
        const int64_t m = d - k0 - n;
        if (m <= 0) continue;
        float* P = w.A + (k0 + n) * d + k0;
        float* A22 = w.A + (k0 + n) * d + k0 + n;
        if (tc) {
            // panel: P <- P * Linv_kk^T
            GPTQ_CUDA_TRY(split_rows(K_SPLIT, P, d, (int)m, n, w.ahi, w.alo, NB, s));
            GPTQ_CUDA_TRY(split_rows(K_SPLIT, LinvK, NB, n, n, w.bhi, w.blo, NB, s));
            GPTQ_CUDA_TRY(tc_gemm_nt(K_TC_PREP, (int)m, n, n, 1.0f, w.ahi, w.alo, w.bhi, w.blo, NB, 0.0f, P, d, false,
                                     w.status, s));
            // trailing: A22 -= P P^T (lower tiles)
            GPTQ_CUDA_TRY(split_rows(K_SPLIT, P, d, (int)m, n, w.ahi, w.alo, NB, s));
            GPTQ_CUDA_TRY(tc_gemm_nt(K_TC_PREP, (int)m, (int)m, n, -1.0f, w.ahi, w.alo, w.ahi, w.alo, NB, 1.0f, A22, d,
                                     true, w.status, s));
        } else {
            GPTQ_CUDA_TRY(sgemm(K_SGEMM_PREP, true, (int)m, n, n, 1.0f, P, d, LinvK, NB, 0.0f, P, d, false, s));
            GPTQ_CUDA_TRY(sgemm(K_SGEMM_PREP, true, (int)m, (int)m, n, -1.0f, P, d, P, d, 1.0f, A22, d, true, s));
        }
    }

    // L^-1 by block rows: X[i,:] = Linv_ii * B[i,:];  B[i+1:, :] -= L[i+1:, i] X[i, :]
    GPTQ_LAUNCH(K_EYE, s, eye_kernel<<<(unsigned)ceil_div(d * d, 256), 256, 0, s>>>(w.Binv, d));
    GPTQ_LAUNCH_CHECK();
    for (int64_t ib = 0; ib < nblk; ++ib) {
        const int64_t i0 = ib * NB;
        const int n = (int)std::min<int64_t>(NB, d - i0);
        const int64_t ncols = i0 + n;
        float* Xi = w.Binv + i0 * d;
        float* LinvI = w.LinvD + ib * NB * NB;
        const int64_t m = d - i0 - n;
        if (tc) {
            // X[i,:] = Linv_ii * X[i,:]: second operand is X[i, 0:ncols]^T (ncols x n)
            GPTQ_CUDA_TRY(split_rows(K_SPLIT, LinvI, NB, n, n, w.ahi, w.alo, NB, s));
            GPTQ_CUDA_TRY(split_cols(K_SPLIT, Xi, d, n, (int)ncols, w.bhi, w.blo, NB, s));
            GPTQ_CUDA_TRY(tc_gemm_nt(K_TC_PREP, n, (int)ncols, n, 1.0f, w.ahi, w.alo, w.bhi, w.blo, NB, 0.0f, Xi, d,
                                     false, w.status, s));
            if (m > 0) {
                GPTQ_CUDA_TRY(split_rows(K_SPLIT, w.A + (i0 + n) * d + i0, d, (int)m, n, w.ahi, w.alo, NB, s));
                GPTQ_CUDA_TRY(split_cols(K_SPLIT, Xi, d, n, (int)ncols, w.bhi, w.blo, NB, s));
                GPTQ_CUDA_TRY(tc_gemm_nt(K_TC_PREP, (int)m, (int)ncols, n, -1.0f, w.ahi, w.alo, w.bhi, w.blo, NB, 1.0f,
                                         w.Binv + (i0 + n) * d, d, false, w.status, s));
            }
        } else {
            GPTQ_CUDA_TRY(sgemm(K_SGEMM_PREP, false, n, (int)ncols, n, 1.0f, LinvI, NB, Xi, d, 0.0f, Xi, d, false, s));
            if (m > 0) {
                GPTQ_CUDA_TRY(sgemm(K_SGEMM_PREP, false, (int)m, (int)ncols, n, -1.0f, w.A + (i0 + n) * d + i0, d, Xi,
                                    d, 1.0f, w.Binv + (i0 + n) * d, d, false, s));
            }
        }
    }

    {
        dim3 grid((unsigned)std::min<int64_t>(ceil_div(d, 256), 64), (unsigned)d);
        GPTQ_LAUNCH(K_SCATTER, s, prep_scatter_kernel<<<grid, 256, 0, s>>>(w.Binv, d, perm, w.rr, U));
        GPTQ_LAUNCH_CHECK();
    }

    int hstatus = 0;
    GPTQ_CUDA_TRY(cudaMemcpyAsync(&hstatus, w.status, sizeof(int), cudaMemcpyDeviceToHost, s));
    GPTQ_CUDA_TRY(cudaStreamSynchronize(s));
    return hstatus;
}

// ------------------------------------------------------------------------------------
// gptq_prepare_noalloc: gptq_prepare for callers that cannot allocate device memory.
//
// Some callers of this library cannot call cudaMalloc for the workspace: a host
// framework that owns every byte of device memory through its own pool and hands out
// nothing extra, or a latency-sensitive path that cannot take cudaMalloc's implicit
// device synchronisation. For them this entry point uses a fixed scratch area compiled
// into the library as a file-scope __device__ array, sized for d <= kNoAllocMaxD.
// Every GPU that loads the library holds this array (about 10.5 MiB) until the process
// exits. The entry point itself allocates nothing: no cudaMalloc, cudaFree or allocating
// library routine.
// ------------------------------------------------------------------------------------
#include <mutex>

namespace gptq {
namespace {

constexpr int64_t kNoAllocMaxD = 1024;

// the workspace gptq_prepare carves for d = kNoAllocMaxD
constexpr size_t kNoAllocBytes = prep_ws_bytes(kNoAllocMaxD);
constexpr int kMaxDevices = 64;

// Host code must not use this name as an address: on the host it is only a stand-in for
// the device symbol. The device address comes from cudaGetSymbolAddress, per device.
static __device__ __align__(256) unsigned char g_prepare_scratch[kNoAllocBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

}  // namespace
}  // namespace gptq

extern "C" int gptq_prepare_noalloc(const float* H, const float* diag_xtx, int64_t d, float damp, int act_order,
                                    float* U, int32_t* perm, uint8_t* dead, void* stream) {
    using namespace gptq;
    if (d <= 0) return GPTQ_ERR_INVALID_ARG;
    if (d > kNoAllocMaxD) return GPTQ_ERR_UNSUPPORTED;
    const size_t need = gptq_prepare_workspace_bytes(d, act_order);
    if (need > kNoAllocBytes) return GPTQ_ERR_UNSUPPORTED;
    int dev = 0;
    GPTQ_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kMaxDevices) return GPTQ_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    {
        // first call on a device: look up this device's copy of the array (once)
        std::lock_guard<std::mutex> lk(g_noalloc_mu);
        if (!g_noalloc_ptr[dev]) {
            void* p = nullptr;
            const cudaError_t e = cudaGetSymbolAddress(&p, g_prepare_scratch);
            if (e != cudaSuccess || p == nullptr) {
                (void)cudaGetLastError();
                return GPTQ_ERR_CUDA;
            }
            g_noalloc_ptr[dev] = p;
        }
        scratch = g_noalloc_ptr[dev];
    }
    // every slab gptq_prepare reads is written by it first (its status word is cleared),
    // so the previous call's contents need no clearing here
    return gptq_prepare(H, diag_xtx, d, damp, act_order, U, perm, dead, scratch, kNoAllocBytes, stream);
}
