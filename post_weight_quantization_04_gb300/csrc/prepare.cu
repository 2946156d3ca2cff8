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
//   A     d*d fp32   reversed, equilibrated Hp -> L below the diagonal blocks (of those
//                    only the inverses are formed, in LinvD or the TF32 splits)
//   Binv  d*d fp32   identity -> L^-1 (lower triangle)
//   LinvD nblk*NB*NB fp32  inverses of L's diagonal blocks
//   TF32 hi/lo splits of the GEMM operands: the panel before its solve and B_k (d x NB);
//   L_kk^-1 twice (even / odd panels); the solved panels L21 of a super-panel (d x SPW,
//   twice: even / odd super-panels) and its block rows of L^-1 (d x SPW), so the next
//   panel can start while the side stream still reads the last ones
//   ddiag d fp32, rr d fp32 (1/sqrt(ddiag)), status int
#include <math.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "sgemm.cuh"
#include "tc_gemm.cuh"

namespace gptq {

namespace {

constexpr int NB = 128;  // panel width of the blocked factorisation
// Panels per super-panel: from kDeferMinD on, the side stream's large rank updates are
// deferred to the end of each super-panel of kSP panels and applied with K = kSP * NB.
#ifndef GPTQ_PREP_SP
#define GPTQ_PREP_SP 4
#endif
constexpr int kSP = GPTQ_PREP_SP;
constexpr int64_t kDeferMinD = 2048;
constexpr int64_t prep_spw(int64_t d) { return (d >= kDeferMinD ? kSP : 1) * (int64_t)NB; }

struct PrepWs {
    float* A;
    float* Binv;
    float* LinvD;
    float* ahi;   // d x NB TF32 splits: the panel before its triangular solve,
    float* alo;
    float* bhi;   //   the block row of the inverse (transposed),
    float* blo;
    float* phi;   //   L21 of the panels of a super-panel (d x SPW), two buffers
    float* plo;   //   (even / odd super-panels),
    float* xhi;   //   the super-panel's block rows of L^-1, transposed (d x SPW),
    float* xlo;
    float* lhi;   // NB x NB: L_kk^-1, two buffers (even / odd panels)
    float* llo;
    float* ddiag;
    float* rr;
    int* status;
    size_t bytes;
};

constexpr size_t align256c(size_t x) { return (x + 255) & ~size_t(255); }

// slab sizes, in carve order; the total is also the size of the allocation-free scratch
constexpr int kPrepSlabs = 16;
constexpr size_t prep_slab(int64_t d, int i) {
    return i < 2 ? sizeof(float) * d * d
         : i == 2 ? sizeof(float) * ((d + NB - 1) / NB) * NB * NB
         : (i == 7 || i == 8) ? sizeof(float) * 2 * d * prep_spw(d)
         : (i == 9 || i == 10) ? sizeof(float) * d * prep_spw(d)
         : i < 11 ? sizeof(float) * d * NB
         : i < 13 ? sizeof(float) * 2 * NB * NB
         : i < 15 ? sizeof(float) * d
         : sizeof(int) * 4;
}
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
    float** f[] = {&w.A, &w.Binv, &w.LinvD, &w.ahi, &w.alo, &w.bhi, &w.blo, &w.phi, &w.plo,
                   &w.xhi, &w.xlo, &w.lhi, &w.llo, &w.ddiag, &w.rr};
    for (int i = 0; i < 15; ++i) *f[i] = reinterpret_cast<float*>(p + off[i]);
    w.status = reinterpret_cast<int*>(p + off[15]);
    w.bytes = off[kPrepSlabs];
    return w;
}

// dead[j] = (H[j][j] == 0); the dead diagonal becomes 1; mean of the fixed diagonal in
// fp64; damped diagonal (rounded to fp32) and its inverse square root in fp32. A diagonal
// entry that is not finite records GPTQ_ERR_NONFINITE.
__global__ void __launch_bounds__(1024) prep_diag_kernel(const float* __restrict__ H, int64_t d, float damp,
                                                        uint8_t* __restrict__ dead, float* __restrict__ ddiag,
                                                        float* __restrict__ rr, int* __restrict__ status) {
    __shared__ double part[32];
    double s = 0.0;
    for (int64_t j = threadIdx.x; j < d; j += blockDim.x) {
        const float h = H[j * d + j];
        if (!isfinite(h)) set_status(status, GPTQ_ERR_NONFINITE);
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
        const float hd = (float)((h == 0.0f ? 1.0 : (double)h) + add);
        ddiag[j] = hd;
        rr[j] = 1.0f / sqrtf(hd);   // fp32 (correctly rounded sqrt and divide)
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
// (fixed, damped diagonal; H read from its upper triangle). An off-diagonal entry that is not
// finite records GPTQ_ERR_NONFINITE.
__global__ void __launch_bounds__(256) prep_gather_kernel(const float* __restrict__ H, int64_t d,
                                                         const int32_t* __restrict__ perm,
                                                         const float* __restrict__ rr, float* __restrict__ A,
                                                         int* __restrict__ status) {
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
        const float h = H[(int64_t)lo * d + hi];
        if (!isfinite(h)) set_status(status, GPTQ_ERR_NONFINITE);
        v = h * rr[a] * rr[b];
    }
    A[i * d + j] = v;
}

// The same without a permutation (perm = identity), four columns per thread with 16-byte
// loads and stores (d % 4 == 0, 16-byte aligned H, A and rr): A[i][j..j+3] comes from the
// group d-4-j .. d-1-j of H's row d-1-i, reversed; only entries on or above H's diagonal
// are read (j + e < i), the diagonal is 1, and the group's entries past A's diagonal
// (never read) are 0. GTH_ROWS rows per CTA.
constexpr int GTH_ROWS = 4;
__global__ void __launch_bounds__(256) prep_gather4_kernel(const float* __restrict__ H, int64_t d,
                                                          const float* __restrict__ rr, float* __restrict__ A,
                                                          int* __restrict__ status) {
    for (int u = 0; u < GTH_ROWS; ++u) {
        const int64_t i = (int64_t)blockIdx.x * GTH_ROWS + u;
        if (i >= d) return;
        const int64_t a = d - 1 - i;
        const float ra = rr[a];
        const float* src = H + a * d;
        float4* dst = reinterpret_cast<float4*>(A + i * d);
        bool bad = false;
        for (int64_t g = threadIdx.x; 4 * g <= i; g += blockDim.x) {
            const int64_t j = 4 * g, c = d - 4 - j;   // H columns c .. c+3 hold A columns j+3 .. j
            float4 h = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (j + 3 <= i) {
                h = *reinterpret_cast<const float4*>(src + c);
            } else {
                if (j + 2 < i) h.y = src[c + 1];
                if (j + 1 < i) h.z = src[c + 2];
                if (j < i) h.w = src[c + 3];
            }
            const float4 r4 = *reinterpret_cast<const float4*>(rr + c);
            float4 o;
            o.x = (j == i) ? 1.0f : h.w * ra * r4.w;
            o.y = (j + 1 == i) ? 1.0f : (j + 1 < i ? h.z * ra * r4.z : 0.0f);
            o.z = (j + 2 == i) ? 1.0f : (j + 2 < i ? h.y * ra * r4.y : 0.0f);
            o.w = (j + 3 == i) ? 1.0f : (j + 3 < i ? h.x * ra * r4.x : 0.0f);
            bad |= (j < i && !isfinite(h.w)) || (j + 1 < i && !isfinite(h.z)) || (j + 2 < i && !isfinite(h.y)) ||
                   (j + 3 < i && !isfinite(h.x));
            dst[g] = o;
        }
        if (bad) set_status(status, GPTQ_ERR_NONFINITE);
    }
}

// Warp-level Cholesky + inverse of a (nb <= 32)-square block held in shared memory. Lane
// r keeps row r of the block (row stride LDS_) in registers. Step k publishes column k of
// the partly reduced block as row k of `lt` (32 x LT_LD floats, 16-byte aligned rows):
// the pivot lt[k][k] and lt[k][i] = L[i][k] * L[k][k] for i > k, which every lane then
// reads with broadcast vector loads. Afterwards lane c forms column c of X = L^-1 by
// forward substitution over the same rows of lt. On return the lower triangle of Xb (row
// stride LDX_) holds L^-1 and XT (32 x LT_LD) holds X transposed (zeros above its diagonal
// and outside nb); L itself is not stored (its users need only L^-1).
constexpr int LT_LD = 36;
template <int LDS_, int LDX_>
__device__ __forceinline__ void chol_inv_32(const float* Sb, float* Xb, float* XT, int nb, float* lt, int* status) {
    const int r = threadIdx.x & 31;
    float dinv[32];
    bool bad = false;
    {
        float a[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) a[c] = (r < nb && c <= r) ? Sb[r * LDS_ + c] : 0.0f;
#pragma unroll
        for (int k = 0; k < 32; ++k) {
            if (k >= nb) break;
            lt[k * LT_LD + r] = a[k];
            __syncwarp();
            const float piv = lt[k * LT_LD + k];
            bad |= !(piv > 0.0f && piv < INFINITY);   // checked once, after the loop
            const float inv = rsqrtf(piv);  // 1 / L[k][k] (hardware approximation, ~2 ulp)
            dinv[k] = inv;
            const float t = a[k] * (inv * inv);  // L[r][k] / L[k][k]
#pragma unroll
            for (int q = (k + 1) >> 2; q < 8; ++q) {
                const float4 v = *reinterpret_cast<const float4*>(lt + k * LT_LD + 4 * q);
                if (4 * q + 0 > k) a[4 * q + 0] = fmaf(-t, v.x, a[4 * q + 0]);
                if (4 * q + 1 > k) a[4 * q + 1] = fmaf(-t, v.y, a[4 * q + 1]);
                if (4 * q + 2 > k) a[4 * q + 2] = fmaf(-t, v.z, a[4 * q + 2]);
                if (4 * q + 3 > k) a[4 * q + 3] = fmaf(-t, v.w, a[4 * q + 3]);
            }
        }
    }
    // a pivot that is not positive and finite: the block is not positive definite; the
    // factorisation goes on with the non-finite values it produces (nothing downstream
    // loops on data) and the call reports the status
    if (bad && r == 0) set_status(status, GPTQ_ERR_NOT_SPD);
    // column r of X: X[k][r] = acc[k] / L[k][k], then acc[i] -= L[i][k] X[k][r] for i > k
    float acc[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) acc[i] = (i == r) ? 1.0f : 0.0f;
#pragma unroll
    for (int k = 0; k < 32; ++k) {
        if (k >= nb) break;
        const float xk = acc[k] * dinv[k];
        acc[k] = xk;
        const float t = xk * dinv[k];
#pragma unroll
        for (int q = (k + 1) >> 2; q < 8; ++q) {
            const float4 v = *reinterpret_cast<const float4*>(lt + k * LT_LD + 4 * q);
            if (4 * q + 0 > k) acc[4 * q + 0] = fmaf(-t, v.x, acc[4 * q + 0]);
            if (4 * q + 1 > k) acc[4 * q + 1] = fmaf(-t, v.y, acc[4 * q + 1]);
            if (4 * q + 2 > k) acc[4 * q + 2] = fmaf(-t, v.z, acc[4 * q + 2]);
            if (4 * q + 3 > k) acc[4 * q + 3] = fmaf(-t, v.w, acc[4 * q + 3]);
        }
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const bool in = i < nb && r < nb && i >= r;
        if (!in) acc[i] = 0.0f;
        if (in) Xb[i * LDX_ + r] = acc[i];
    }
#pragma unroll
    for (int q = 0; q < 8; ++q)
        *reinterpret_cast<float4*>(XT + r * LT_LD + 4 * q) = make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2],
                                                                         acc[4 * q + 3]);
    __syncwarp();  // lt is reused by the next call
}

// named barrier 1: warps 1-3 hand the updated next diagonal block to warp 0
__device__ __forceinline__ void bar_arrive_diag() { asm volatile("bar.arrive 1, 128;" ::: "memory"); }
__device__ __forceinline__ void bar_sync_diag() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// (ti, tj) of the t-th 4 x 4 tile of a lower triangle, row by row
__device__ __forceinline__ void tri_tile(int t, int& ti, int& tj) {
    int i = (int)((sqrtf(8.0f * (float)t + 1.0f) - 1.0f) * 0.5f);
    while ((i + 1) * (i + 2) / 2 <= t) ++i;
    while (i * (i + 1) / 2 > t) --i;
    ti = i;
    tj = t - i * (i + 1) / 2;
}

// One CTA factors the diagonal block A[k0:k0+n, k0:k0+n] = L L^T and forms L^-1 (lower,
// NB x NB, zeros above): optionally written to Linv, and as its TF32 split to Lhi/Llo
// (its zero upper triangle only when split_upper; otherwise the buffer must hold zeros
// there already).
// A is only read: the callers need L^-1 alone. A non-positive or non-finite pivot records
// GPTQ_ERR_NOT_SPD (the kernel still finishes; its outputs are then not finite).
//
// Blocked by 32 columns inside shared memory. For each 32-column sub-panel b:
//   1. warp 0: L_bb and X_bb = L_bb^-1 (chol_inv_32)
//   2. the panel below it, L21 = A21 X_bb^T (kept also transposed in Lt), and the block
//      row of the inverse left of the diagonal, X[b, :b] = X_bb B[b, :b]
//   3. the trailing update A22 -= L21 L21^T (its next diagonal block first, by warps 1-3,
//      then factored by warp 0) and the inverse's right-looking update
//      B[below, :b+32] -= L21 X[b, :b+32]
// (B, the right-hand side of L X = I, lives in X's storage until it is overwritten.)
// All products are register tiles over shared memory, read with 16-byte loads.
constexpr int POTRF_LDS = NB + 1;   // row stride of the block (odd: conflict-free columns)
constexpr int POTRF_LDX = NB + 4;   // row stride of L^-1 and of Lt (16-byte rows)
constexpr size_t potrf_smem_bytes() {
    return sizeof(float) * ((size_t)NB * POTRF_LDS + (size_t)NB * POTRF_LDX + 32 * (size_t)POTRF_LDX + 2 * 32 * LT_LD);
}
__global__ void __launch_bounds__(512) potrf_diag_kernel(const float* __restrict__ A, int64_t lda, int64_t k0, int n,
                                                        float* __restrict__ Linv, float* __restrict__ Lhi,
                                                        float* __restrict__ Llo, int split_upper,
                                                        int* __restrict__ status) {
    extern __shared__ __align__(16) float sm[];
    constexpr int LD = POTRF_LDS, LDX = POTRF_LDX;
    float* S = sm;                   // NB x LD: the block (lower triangle), updated in place
    float* X = S + NB * LD;          // NB x LDX: B, then L^-1
    float* Lt = X + NB * LDX;        // 32 x LDX: the current panel of L, transposed
    float* XT = Lt + 32 * LDX;       // 32 x LT_LD: X_bb transposed
    float* lt = XT + 32 * LT_LD;     // 32 x LT_LD: chol_inv_32 scratch
    const int tid = threadIdx.x;
    pdl_wait();
    pdl_trigger();

    {
        // the lower triangle in 16-byte pieces, the lanes of a warp on 32 consecutive rows
        // (conflict-free stores into the odd-stride block); all loads of a thread in flight
        // at once
        const bool vec = ((lda & 3) == 0) && ((k0 & 3) == 0) && ((reinterpret_cast<uintptr_t>(A) & 15) == 0);
        float4 v[NB * NB / 4 / 512];
#pragma unroll
        for (int u = 0; u < NB * NB / 4 / 512; ++u) {
            const int idx = tid + 512 * u;
            const int i = idx & (NB - 1), j4 = (idx >> 7) << 2;
            float4 x = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (i < n && j4 <= i) {
                const float* src = A + (k0 + i) * lda + k0 + j4;
                if (vec && j4 + 3 < n) {
                    x = *reinterpret_cast<const float4*>(src);
                } else {
                    x.x = src[0];
                    if (j4 + 1 < n) x.y = src[1];
                    if (j4 + 2 < n) x.z = src[2];
                    if (j4 + 3 < n) x.w = src[3];
                }
                if (j4 + 1 > i) x.y = 0.0f;
                if (j4 + 2 > i) x.z = 0.0f;
                if (j4 + 3 > i) x.w = 0.0f;
            }
            v[u] = x;
        }
#pragma unroll
        for (int u = 0; u < NB * NB / 4 / 512; ++u) {
            const int idx = tid + 512 * u;
            float* d = S + (idx & (NB - 1)) * LD + ((idx >> 7) << 2);
            d[0] = v[u].x;
            d[1] = v[u].y;
            d[2] = v[u].z;
            d[3] = v[u].w;
        }
        for (int idx = tid; idx < NB * LDX / 4; idx += 512)
            reinterpret_cast<float4*>(X)[idx] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
    __syncthreads();
    if (tid < 32) chol_inv_32<LD, LDX>(S, X, XT, min(32, n), lt, status);

    // the diagonal block of sub-panel b is factored (warp 0) before the iteration starts:
    // for b = 0 above, for the next ones at the end of the previous iteration
    for (int b = 0; b < n; b += 32) {
        __syncthreads();
        const int rb = b + 32, m = max(0, n - rb);
        const int tm = (m + 3) >> 2;       // 4-row tiles below the sub-panel
        // ---- 2. panel L21 = A21 X_bb^T (2 x 4 tiles: up to 384 threads, each a short
        //      chain on the critical path), and X[b, :b] = X_bb B[b, :b] (4 x 4 tiles) ----
        {
            const int P = 8 * ((m + 1) >> 1), Q = 8 * (b >> 2);
            float acc[4][4];
            int kind = -1, r0 = 0, c0 = 0;
            const int t = tid;
            if (t < P) {
                kind = 0;
                r0 = rb + 2 * (t >> 3);
                c0 = 4 * (t & 7);
#pragma unroll
                for (int u = 0; u < 2; ++u)
#pragma unroll
                    for (int v = 0; v < 4; ++v) acc[u][v] = 0.0f;
#pragma unroll 4
                for (int k = 0; k < 32; ++k) {
                    const float4 x4 = *reinterpret_cast<const float4*>(XT + k * LT_LD + c0);
                    float ar[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) ar[u] = (r0 + u < n) ? S[(r0 + u) * LD + b + k] : 0.0f;
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        acc[u][0] = fmaf(ar[u], x4.x, acc[u][0]);
                        acc[u][1] = fmaf(ar[u], x4.y, acc[u][1]);
                        acc[u][2] = fmaf(ar[u], x4.z, acc[u][2]);
                        acc[u][3] = fmaf(ar[u], x4.w, acc[u][3]);
                    }
                }
            } else if (t < P + Q) {
                kind = 1;
                const int q = t - P;
                r0 = b + 4 * (q & 7);
                c0 = 4 * (q >> 3);
#pragma unroll
                for (int u = 0; u < 4; ++u)
#pragma unroll
                    for (int v = 0; v < 4; ++v) acc[u][v] = 0.0f;
#pragma unroll 4
                for (int k = 0; k < 32; ++k) {
                    const float4 a4 = *reinterpret_cast<const float4*>(XT + k * LT_LD + (r0 - b));
                    const float4 b4 = *reinterpret_cast<const float4*>(X + (b + k) * LDX + c0);
                    const float ar[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        acc[u][0] = fmaf(ar[u], b4.x, acc[u][0]);
                        acc[u][1] = fmaf(ar[u], b4.y, acc[u][1]);
                        acc[u][2] = fmaf(ar[u], b4.z, acc[u][2]);
                        acc[u][3] = fmaf(ar[u], b4.w, acc[u][3]);
                    }
                }
            }
            __syncthreads();  // X[b, :b] is read above before it is overwritten below
            if (kind == 0) {
                // L21 is needed only transposed, in Lt (its rows of S are never read again)
#pragma unroll
                for (int v = 0; v < 4; ++v)
                    *reinterpret_cast<float2*>(Lt + (c0 + v) * LDX + r0) =
                        make_float2(r0 < n ? acc[0][v] : 0.0f, r0 + 1 < n ? acc[1][v] : 0.0f);
            } else if (kind == 1) {
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if (r0 + u < n)
                        *reinterpret_cast<float4*>(X + (r0 + u) * LDX + c0) =
                            make_float4(acc[u][0], acc[u][1], acc[u][2], acc[u][3]);
            }
        }
        if (m <= 0) break;
        __syncthreads();
        // ---- 3. A22 -= L21 L21^T (lower tiles) and B[below, :b+32] -= L21 X[b, :b+32] ----
        // Warps 1-3 update the next diagonal block first (4 x 4 tiles, one per thread) and
        // hand it to warp 0 through a named barrier; warp 0 factors it while the 12 warps
        // outside its SM sub-partition (warp % 4 != 0) do the rest in 8 x 4 tiles (three
        // 16-byte loads per 32 FMAs, so the shared-memory traffic leaves room for the
        // factorisation); warps 4, 8 and 12 stay idle so the latency-bound factorisation
        // has its issue slots to itself.
        if (tid < 32) {
            bar_sync_diag();   // warps 1-3 have updated the next diagonal block
            chol_inv_32<LD, LDX>(S + rb * LD + rb, X + rb * LDX + rb, XT, min(32, m), lt, status);
        } else if ((tid >> 5) & 3) {
            const int w = tid >> 5, p = (w - 1 - (w >> 2)) * 32 + (tid & 31);  // 0 .. 383
            if (w < 4) {
                // warps 1-3 (one per other SM sub-partition): the next diagonal block first,
                // A22' -= L21' L21'^T in 4 x 4 tiles (at most 36: one per thread)
                const int D = min(tm, 8), Td = D * (D + 1) / 2;
                if (p < Td) {
                    const int t = p;
                    int ti, tj;
                    tri_tile(t, ti, tj);
                    const int r0 = rb + 4 * ti, c0 = rb + 4 * tj;
                    float acc[4][4];
#pragma unroll
                    for (int u = 0; u < 4; ++u)
#pragma unroll
                        for (int v = 0; v < 4; ++v) acc[u][v] = 0.0f;
#pragma unroll 4
                    for (int k = 0; k < 32; ++k) {
                        const float4 a4 = *reinterpret_cast<const float4*>(Lt + k * LDX + r0);
                        const float4 b4 = *reinterpret_cast<const float4*>(Lt + k * LDX + c0);
                        const float ar[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            acc[u][0] = fmaf(ar[u], b4.x, acc[u][0]);
                            acc[u][1] = fmaf(ar[u], b4.y, acc[u][1]);
                            acc[u][2] = fmaf(ar[u], b4.z, acc[u][2]);
                            acc[u][3] = fmaf(ar[u], b4.w, acc[u][3]);
                        }
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u)
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            if (r0 + u < n && c0 + v <= r0 + u) S[(r0 + u) * LD + c0 + v] -= acc[u][v];
                }
                bar_arrive_diag();
            }
            const int t8 = (m + 7) >> 3;                  // 8-row tiles below the sub-panel
            // SYRK: 8 x 8 blocks below the next diagonal block, each as two 8 x 4 tiles
            const int Ts = 2 * max(0, t8 * (t8 + 1) / 2 - 10);
            const int nbt = (b + 32) >> 2, Tb = t8 * nbt;  // inverse update: 8 x 4 tiles
            for (int t = p; t < Ts + Tb; t += 384) {
                int r0, c0;
                const float* bsrc;
                if (t < Ts) {
                    int ti, tj;
                    tri_tile((t >> 1) + 10, ti, tj);   // triangle rows 0-3 are the diagonal block
                    r0 = rb + 8 * ti;
                    c0 = rb + 8 * tj + 4 * (t & 1);
                    bsrc = Lt + c0;
                } else {
                    const int q = t - Ts;
                    r0 = rb + 8 * (q / nbt);
                    c0 = 4 * (q % nbt);
                    bsrc = X + b * LDX + c0;
                }
                float acc[8][4];
#pragma unroll
                for (int u = 0; u < 8; ++u)
#pragma unroll
                    for (int v = 0; v < 4; ++v) acc[u][v] = 0.0f;
#pragma unroll 2
                for (int k = 0; k < 32; ++k) {
                    const float4 a0 = *reinterpret_cast<const float4*>(Lt + k * LDX + r0);
                    const float4 a1 = *reinterpret_cast<const float4*>(Lt + k * LDX + r0 + 4);
                    const float4 b0 = *reinterpret_cast<const float4*>(bsrc + k * LDX);
                    const float ar[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        acc[u][0] = fmaf(ar[u], b0.x, acc[u][0]);
                        acc[u][1] = fmaf(ar[u], b0.y, acc[u][1]);
                        acc[u][2] = fmaf(ar[u], b0.z, acc[u][2]);
                        acc[u][3] = fmaf(ar[u], b0.w, acc[u][3]);
                    }
                }
                if (t < Ts) {
#pragma unroll
                    for (int u = 0; u < 8; ++u)
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            if (r0 + u < n && c0 + v <= r0 + u) S[(r0 + u) * LD + c0 + v] -= acc[u][v];
                } else {
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        if (r0 + u < n) {
                            float4* xp = reinterpret_cast<float4*>(X + (r0 + u) * LDX + c0);
                            float4 xv = *xp;
                            xv.x -= acc[u][0];
                            xv.y -= acc[u][1];
                            xv.z -= acc[u][2];
                            xv.w -= acc[u][3];
                            *xp = xv;
                        }
                }
            }
        }
    }
    __syncthreads();

#pragma unroll 2
    for (int idx = tid; idx < NB * NB / 4; idx += 512) {
        const int i = idx >> 5, j4 = (idx & 31) << 2;
        float4 v = *reinterpret_cast<const float4*>(X + i * LDX + j4);
        if (i >= n) v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (j4 + 0 > i || j4 + 0 >= n) v.x = 0.0f;
        if (j4 + 1 > i || j4 + 1 >= n) v.y = 0.0f;
        if (j4 + 2 > i || j4 + 2 >= n) v.z = 0.0f;
        if (j4 + 3 > i || j4 + 3 >= n) v.w = 0.0f;
        if (Linv) *reinterpret_cast<float4*>(Linv + 4 * idx) = v;
        // TF32 split for the tensor-core products that use L_kk^-1; the groups of four
        // entirely above the diagonal are zero and, unless split_upper, already zero in
        // the buffer (written by an earlier call on it)
        if (Lhi && (split_upper || j4 <= i)) {
            float4 h;
            h.x = __uint_as_float(__float_as_uint(v.x) & 0xFFFFE000u);
            h.y = __uint_as_float(__float_as_uint(v.y) & 0xFFFFE000u);
            h.z = __uint_as_float(__float_as_uint(v.z) & 0xFFFFE000u);
            h.w = __uint_as_float(__float_as_uint(v.w) & 0xFFFFE000u);
            *reinterpret_cast<float4*>(Lhi + 4 * idx) = h;
            *reinterpret_cast<float4*>(Llo + 4 * idx) = make_float4(v.x - h.x, v.y - h.y, v.z - h.z, v.w - h.w);
        }
    }
}

__global__ void eye_kernel(float* __restrict__ B, int64_t d) {
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx < d * d) B[idx] = (idx / d == idx % d) ? 1.0f : 0.0f;
}

// The identity with 16-byte stores (d % 4 == 0, B 16-byte aligned): grid-stride over the
// d*d/4 groups of four, one row per block of d/4 groups.
__global__ void __launch_bounds__(256) eye4_kernel(float* __restrict__ B, int64_t d) {
    const int64_t q = d >> 2, total = d * q;
    for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < total; g += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i = g / q, c = (g - i * q) << 2;
        float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (i >= c && i < c + 4) {
            const int e = (int)(i - c);
            v.x = e == 0 ? 1.0f : 0.0f;
            v.y = e == 1 ? 1.0f : 0.0f;
            v.z = e == 2 ? 1.0f : 0.0f;
            v.w = e == 3 ? 1.0f : 0.0f;
        }
        reinterpret_cast<float4*>(B)[g] = v;
    }
}

// U[i][j] = (i <= j) ? Linv[d-1-i][d-1-j] * rr[perm[j]] : 0, four columns per thread with
// 16-byte loads and stores (d % 4 == 0, 16-byte aligned bases): the four columns j..j+3 of
// U's row i are the 16-byte group d-4-j .. d-1-j of Linv's row d-1-i, reversed. SCR_ROWS
// rows per CTA; the groups left of the diagonal are zeros and read nothing.
constexpr int SCR_ROWS = 4;
__global__ void __launch_bounds__(256) prep_scatter4_kernel(const float* __restrict__ Binv, int64_t d,
                                                           const int32_t* __restrict__ perm,
                                                           const float* __restrict__ rr, float* __restrict__ U) {
    const int64_t q = d >> 2;
    for (int u = 0; u < SCR_ROWS; ++u) {
        const int64_t i = (int64_t)blockIdx.x * SCR_ROWS + u;
        if (i >= d) return;
        const float* src = Binv + (d - 1 - i) * d;
        float4* dst = reinterpret_cast<float4*>(U + i * d);
        for (int64_t g = threadIdx.x; g < q; g += blockDim.x) {
            const int64_t j = g << 2;
            float4 o = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (j + 3 >= i) {
                const float4 b = *reinterpret_cast<const float4*>(src + (d - 4 - j));
                const int4 p = *reinterpret_cast<const int4*>(perm + j);
                o.x = (j + 0 >= i) ? b.w * rr[p.x] : 0.0f;
                o.y = (j + 1 >= i) ? b.z * rr[p.y] : 0.0f;
                o.z = (j + 2 >= i) ? b.y * rr[p.z] : 0.0f;
                o.w = (j + 3 >= i) ? b.x * rr[p.w] : 0.0f;
            }
            dst[g] = o;
        }
    }
}

// U[i][j] = (i <= j) ? Linv[d-1-i][d-1-j] * rr[perm[j]] : 0 (any d)
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

namespace gptq {
namespace {

// Streams and events for the two-stream factorisation: one set per (device, caller stream)
// (up to kSetsPerDevice per device; beyond that, caller streams share sets), created on
// first use and kept for the life of the process. Calls on different caller streams run on
// different sets, so their factorisations can overlap on the GPU; a set's mutex is held for
// the whole call, so calls that share a set take its streams in turn (their work is then
// ordered on the set's streams, which is still correct).
#ifndef GPTQ_CHAIN_SMS
#define GPTQ_CHAIN_SMS 32
#endif
constexpr int kChainSMs = GPTQ_CHAIN_SMS;
constexpr int kMaxPrepDevices = 64;
constexpr int kSetsPerDevice = 8;
struct PrepConcurrency {
    std::mutex mu;
    cudaStream_t owner = nullptr;   // the caller stream this set serves
    bool used = false;
    bool ready = false;
    cudaStream_t crit = nullptr, side = nullptr;
    cudaEvent_t fork = nullptr, trsm = nullptr, rest = nullptr, rest_far = nullptr, side_done[2] = {nullptr, nullptr},
                far_done[2] = {nullptr, nullptr}, join_side = nullptr, join_crit = nullptr;
};
PrepConcurrency g_conc[kMaxPrepDevices][kSetsPerDevice];
std::mutex g_conc_mu;   // guards the owner assignment of the sets

// The set for caller stream s on device dev: the one it used before, else a free one, else
// one shared by hash.
PrepConcurrency& conc_for(int dev, cudaStream_t s) {
    std::lock_guard<std::mutex> lk(g_conc_mu);
    PrepConcurrency* sets = g_conc[dev];
    for (int i = 0; i < kSetsPerDevice; ++i)
        if (sets[i].used && sets[i].owner == s) return sets[i];
    for (int i = 0; i < kSetsPerDevice; ++i)
        if (!sets[i].used) {
            sets[i].used = true;
            sets[i].owner = s;
            return sets[i];
        }
    return sets[(reinterpret_cast<uintptr_t>(s) >> 4) % kSetsPerDevice];
}

// The chain stream takes the device's greatest priority (its kernels are the critical path
// of the call); the side stream takes the caller stream's priority, so a caller that runs
// one factorisation ahead of other work (a high-priority stream) gets its bulk updates
// ahead of that work too, and a default-priority caller gets the default.
cudaError_t conc_init(PrepConcurrency& c, cudaStream_t caller) {
    if (c.ready) return cudaSuccess;
    int least = 0, greatest = 0, pc = 0;
    cudaError_t e = cudaDeviceGetStreamPriorityRange(&least, &greatest);
    if (e == cudaSuccess) e = cudaStreamGetPriority(caller, &pc);
    if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&c.crit, cudaStreamNonBlocking, greatest);
    if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&c.side, cudaStreamNonBlocking, pc);
    cudaEvent_t* evs[] = {&c.fork,          &c.trsm,        &c.rest,        &c.rest_far,  &c.side_done[0],
                          &c.side_done[1], &c.far_done[0], &c.far_done[1], &c.join_side, &c.join_crit};
    for (cudaEvent_t* ev : evs)
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    if (e == cudaSuccess) c.ready = true;
    return e;
}

int check_args(const float* H, const float* diag_xtx, int64_t d, float damp, int act_order, const float* U,
               const int32_t* perm, const uint8_t* dead, const void* ws, size_t ws_bytes) {
    if (d <= 0 || d > (1 << 20) || !H || !U || !perm || !dead || !ws) return GPTQ_ERR_INVALID_ARG;
    if (act_order && !diag_xtx) return GPTQ_ERR_INVALID_ARG;
    if (!(damp >= 0.0f) || !isfinite(damp)) return GPTQ_ERR_INVALID_ARG;
    if (ws_bytes < carve(nullptr, d).bytes) return GPTQ_ERR_WORKSPACE;
    return GPTQ_OK;
}

int prepare_impl(const float* H, const float* diag_xtx, int64_t d, float damp, int act_order, float* U,
                 int32_t* perm, uint8_t* dead, void* ws, size_t ws_bytes, void* stream_, PrepConcurrency* conc) {
    const int arg = check_args(H, diag_xtx, d, damp, act_order, U, perm, dead, ws, ws_bytes);
    if (arg != GPTQ_OK) return arg;
    PrepWs w = carve(ws, d);
    cudaStream_t s = static_cast<cudaStream_t>(stream_);

    GPTQ_CUDA_TRY(cudaMemsetAsync(w.status, 0, sizeof(int), s));
    GPTQ_LAUNCH(K_PREP_DIAG, s, prep_diag_kernel<<<1, 1024, 0, s>>>(H, d, damp, dead, w.ddiag, w.rr, w.status));
    GPTQ_LAUNCH_CHECK();
    const unsigned g1 = (unsigned)ceil_div(d, 256);
    if (act_order)
        GPTQ_LAUNCH(K_PREP_PERM, s, prep_perm_kernel<<<g1, 256, 0, s>>>(diag_xtx, d, perm));
    else
        GPTQ_LAUNCH(K_PREP_PERM, s, iota_kernel<<<g1, 256, 0, s>>>(perm, d));
    GPTQ_LAUNCH_CHECK();
    if (!act_order && d % 4 == 0 && ((reinterpret_cast<uintptr_t>(H) | reinterpret_cast<uintptr_t>(w.A)) % 16 == 0)) {
        GPTQ_LAUNCH(K_PREP_GATHER, s, prep_gather4_kernel<<<(unsigned)ceil_div(d, GTH_ROWS), 256, 0, s>>>(
                                          H, d, w.rr, w.A, w.status));
        GPTQ_LAUNCH_CHECK();
    } else {
        dim3 grid((unsigned)ceil_div(d, 32), (unsigned)ceil_div(d, 8));
        GPTQ_LAUNCH(K_PREP_GATHER, s, prep_gather_kernel<<<grid, 256, 0, s>>>(H, d, perm, w.rr, w.A, w.status));
        GPTQ_LAUNCH_CHECK();
    }

    const size_t potrf_smem = potrf_smem_bytes();
    GPTQ_CUDA_TRY(cudaFuncSetAttribute(potrf_diag_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)potrf_smem));

    // The trailing contractions run on the tensor cores (3xTF32, operands split into
    // TF32 hi/lo) when every matrix row is 16-byte aligned, else on the FFMA GEMM.
    const bool tc = (d % 4 == 0) && tc_gemm_nt_ok(w.A, d);

    const int64_t nblk = ceil_div(d, NB);
    const bool vec4 = (d % 4 == 0) && ((reinterpret_cast<uintptr_t>(w.Binv) | reinterpret_cast<uintptr_t>(U) |
                                        reinterpret_cast<uintptr_t>(perm)) % 16 == 0);
    auto launch_eye = [&](cudaStream_t st) -> int {
        if (vec4) {
            const unsigned g = (unsigned)std::min<int64_t>(ceil_div(d * d / 4, 256), (int64_t)device_sm_count() * 8);
            GPTQ_LAUNCH(K_EYE, st, eye4_kernel<<<g, 256, 0, st>>>(w.Binv, d));
        } else {
            GPTQ_LAUNCH(K_EYE, st, eye_kernel<<<(unsigned)ceil_div(d * d, 256), 256, 0, st>>>(w.Binv, d));
        }
        GPTQ_LAUNCH_CHECK();
        return GPTQ_OK;
    };
    if (!tc || !conc) {
        const int rc = launch_eye(s);
        if (rc != GPTQ_OK) return rc;
    }
    if (tc) {
        // Blocked right-looking Cholesky of A (lower) with the block-row inverse step of
        // L^-1 interleaved, in two streams. The critical chain (stream `cs`) is
        //   potrf(k) -> panel solve L21 = P L_kk^-T -> SYRK of the next panel's columns
        //   -> potrf(k+1) ...
        // while the side stream (`ss`) applies the rest of panel k's SYRK and the inverse
        // step X_k = L_kk^-1 B_k, B[k+1:, :] -= L21 X_k, reading panel k's TF32 splits.
        // The splits of L21 and L_kk^-1 alternate between two buffers by panel parity; the
        // chain waits for the side stream to finish panel k-2 before it overwrites them.
        // kChainSMs SMs are kept for the chain, the rest for the side stream.
        const bool two = conc != nullptr;
        cudaStream_t cs = two ? conc->crit : s, ss = two ? conc->side : s;
        auto record = [&](cudaEvent_t e, cudaStream_t st) -> cudaError_t {
            return two ? cudaEventRecord(e, st) : cudaSuccess;
        };
        auto wait = [&](cudaStream_t st, cudaEvent_t e) -> cudaError_t {
            return two ? cudaStreamWaitEvent(st, e, 0) : cudaSuccess;
        };
        if (two) {
            GPTQ_CUDA_TRY(record(conc->fork, s));
            GPTQ_CUDA_TRY(wait(cs, conc->fork));
            GPTQ_CUDA_TRY(wait(ss, conc->fork));
            // B = I (the right-hand side of L X = I) is first read by the side stream
            const int rc = launch_eye(ss);
            if (rc != GPTQ_OK) return rc;
        }
        // the SMs are split between the streams: persistent CTAs of one stream would
        // otherwise hold SMs that the other's next kernel waits for
        GemmOpts side_opts, chain_opts;
        side_opts.max_ctas = two ? std::max(1, device_sm_count() - kChainSMs) : 0;
        chain_opts.max_ctas = two ? kChainSMs : 0;
        chain_opts.narrow_ok = true;   // the factorisation chain is latency-bound
        // Programmatic dependent launch only where the previous item in the stream is one
        // of these kernels (not an event wait): cs_k / ss_k say whether it is.
        bool cs_k = !two, ss_k = false;
        auto waited = [&](cudaStream_t st) {
            if (st == cs) cs_k = false;
            if (st == ss) ss_k = false;
        };
        // Super-panels. L21 of each panel is split into column block j (= its index in the
        // super-panel) of the super-panel's buffer phi/plo (row stride SPW; buffer row
        // r = global row - (sp0 + NB), so panel j's L21 starts at row NB * j), and each
        // block row X_k of L^-1 into column block j of xhi/xlo (transposed, row stride SPW).
        // Inside a super-panel the side stream updates only the super-panel's own columns
        // (of A and of B = L^-1's right-hand side); at its end it updates everything past
        // it with the errors of all its panels at once (K = SPW). With SPW = NB this is the
        // plain one-panel-at-a-time schedule.
        const int64_t SPW = prep_spw(d);
        const int SP = (int)(SPW / NB);
        for (int64_t kb = 0; kb < nblk; ++kb) {
            const int64_t k0 = kb * NB;
            const int n = (int)std::min<int64_t>(NB, d - k0);
            const int64_t m = d - k0 - n, ncols = k0 + n;
            const int nn = (int)std::min<int64_t>(NB, m);  // width of the next panel
            const int par = (int)(kb & 1);
            const int64_t sp = kb / SP, j = kb % SP;
            const int64_t sp0 = sp * SPW, sp_end = std::min<int64_t>(d, sp0 + SPW);
            const bool sp_last = (k0 + n == sp_end);   // last panel of its super-panel
            const int spar = (int)(sp & 1);
            float* lhi = w.lhi + par * NB * NB;
            float* llo = w.llo + par * NB * NB;
            float* shi = w.phi + spar * d * SPW;   // this super-panel's L21 splits
            float* slo = w.plo + spar * d * SPW;
            float* Lhi = shi + (NB * j) * SPW + NB * j;   // this panel's L21 split (m x n)
            float* Llo = slo + (NB * j) * SPW + NB * j;
            // rows at or below sp_end of all the super-panel's L21 (the deferred updates' operand)
            float* Ehi = shi + (SPW - NB) * SPW;
            float* Elo = slo + (SPW - NB) * SPW;
            if (two && kb >= 2) {   // L_kk^-1 buffer par: read by the side stream's panel kb-2
                GPTQ_CUDA_TRY(wait(cs, conc->side_done[par]));
                waited(cs);
            }
            if (two && j == 0 && sp >= 2) {   // super-panel buffer spar: read up to the end of sp-2
                GPTQ_CUDA_TRY(wait(cs, conc->far_done[spar]));
                waited(cs);
            }
            if (cs_k) {
                cudaError_t le = cudaSuccess;
                // each of the two L_kk^-1 buffers gets its zero upper triangle on its first use
                GPTQ_LAUNCH(K_POTRF, cs, le = launch_pdl(potrf_diag_kernel, dim3(1), dim3(512), potrf_smem, cs,
                                                         (const float*)w.A, d, k0, n, (float*)nullptr, lhi, llo,
                                                         (int)(kb < 2), w.status));
                GPTQ_CUDA_TRY(le);
            } else {
                GPTQ_LAUNCH(K_POTRF, cs, potrf_diag_kernel<<<1, 512, potrf_smem, cs>>>(w.A, d, k0, n, nullptr, lhi,
                                                                                      llo, (int)(kb < 2), w.status));
            }
            GPTQ_LAUNCH_CHECK();
            cs_k = true;
            float* P = w.A + (k0 + n) * d + k0;
            if (m > 0) {
                GemmOpts l21 = chain_opts;  // L21 split for the trailing updates and the inverse step
                l21.hi = Lhi;
                l21.lo = Llo;
                l21.ld = SPW;
                l21.mode = 1;
                l21.pdl = true;
                // the panel's split: for panel 0 here; for the others it was written by the
                // previous panel's SYRK of these columns (its rows below the diagonal block)
                if (kb == 0) GPTQ_CUDA_TRY(split_rows(K_SPLIT, P, d, (int)m, n, w.ahi, w.alo, NB, cs, true));
                GPTQ_CUDA_TRY(tc_gemm_nt(K_TC_CHAIN, (int)m, n, n, 1.0f, w.ahi, w.alo, lhi, llo, NB, 0.0f, P, d,
                                         false, w.status, cs, l21));
                GPTQ_CUDA_TRY(record(two ? conc->trsm : nullptr, cs));
                // the next panel's columns; the side stream's updates wrote them too: inside
                // a super-panel the previous panel's update of the super-panel's columns (or
                // the first part of the previous super-panel's deferred update), for the first
                // panel of the next super-panel the second part of that deferred update
                if (two && kb >= 1 && (!sp_last || sp >= 1)) {
                    GPTQ_CUDA_TRY(wait(cs, sp_last ? conc->rest_far : conc->rest));
                    waited(cs);
                }
                GemmOpts strip = chain_opts;
                strip.pdl = cs_k;
                strip.hi = w.ahi;   // rows below the next diagonal block = the next panel, split
                strip.lo = w.alo;
                strip.ld = NB;
                strip.mode = 1;
                strip.row0 = nn;
                // inside the super-panel: this panel's L21 (K = n); at its end the next panel
                // starts a new super-panel and takes all of this one's panels (K = SPW)
                const int ks = sp_last ? (int)SPW : n;
                const float* sh = sp_last ? Ehi : Lhi;
                const float* sl = sp_last ? Elo : Llo;
                GPTQ_CUDA_TRY(tc_gemm_nt(K_TC_CHAIN, (int)m, nn, ks, -1.0f, sh, sl, sh, sl, (int)SPW, 1.0f,
                                         w.A + (k0 + n) * d + k0 + n, d, true, w.status, cs, strip));
                cs_k = true;
            } else {
                GPTQ_CUDA_TRY(record(two ? conc->trsm : nullptr, cs));
            }
            GPTQ_CUDA_TRY(wait(ss, two ? conc->trsm : nullptr));
            waited(ss);
            auto side_gemm = [&](int M, int N, int K, const float* ah, const float* al, const float* bh,
                                 const float* bl, float* C, bool lower) -> cudaError_t {
                if (M <= 0 || N <= 0) return cudaSuccess;
                GemmOpts o = side_opts;
                o.pdl = ss_k;
                const cudaError_t e = tc_gemm_nt(K_TC_PREP, M, N, K, -1.0f, ah, al, bh, bl, (int)SPW, 1.0f, C, d,
                                                 lower, w.status, ss, o);
                if (e == cudaSuccess) ss_k = true;
                return e;
            };
            if (m > 0 && !sp_last) {
                // A[c0:, c0:sp_end] -= L21[nn:] L21[nn : sp_end-k0-n]^T (the super-panel's own
                // columns past the next panel)
                const int64_t c0 = k0 + n + nn;
                GPTQ_CUDA_TRY(side_gemm((int)(d - c0), (int)(sp_end - c0), n, Lhi + nn * SPW, Llo + nn * SPW,
                                        Lhi + nn * SPW, Llo + nn * SPW, w.A + c0 * (d + 1), true));
            }
            if (m > 0 && sp_last) {
                // deferred: first the next super-panel's columns past its first panel (the
                // chain needs them next), then everything past the next super-panel
                const int64_t c0 = sp_end + nn, c1 = std::min<int64_t>(d, sp_end + SPW);
                GPTQ_CUDA_TRY(side_gemm((int)(d - c0), (int)(c1 - c0), (int)SPW, Ehi + nn * SPW, Elo + nn * SPW,
                                        Ehi + nn * SPW, Elo + nn * SPW, w.A + c0 * (d + 1), true));
                GPTQ_CUDA_TRY(record(two ? conc->rest : nullptr, ss));
                const int64_t rb = c1 - sp_end;   // rows of E from c1 on
                GPTQ_CUDA_TRY(side_gemm((int)(d - c1), (int)(d - c1), (int)SPW, Ehi + rb * SPW, Elo + rb * SPW,
                                        Ehi + rb * SPW, Elo + rb * SPW, w.A + c1 * (d + 1), true));
                GPTQ_CUDA_TRY(record(two ? conc->rest_far : nullptr, ss));
            } else {
                GPTQ_CUDA_TRY(record(two ? conc->rest : nullptr, ss));
            }
            // X_k = L_kk^-1 B_k over the super-panel's columns (B_k is zero from ncols on)
            const int64_t xn = sp_end;
            float* Xi = w.Binv + k0 * d;
            GemmOpts xt = side_opts;  // X_k^T split for the inverse's trailing updates
            xt.hi = w.xhi + NB * j;
            xt.lo = w.xlo + NB * j;
            xt.ld = SPW;
            xt.mode = 2;
            xt.pdl = true;
            GPTQ_CUDA_TRY(split_cols(K_SPLIT, Xi, d, n, (int)xn, w.bhi, w.blo, NB, ss, ss_k));
            GPTQ_CUDA_TRY(tc_gemm_nt(K_TC_PREP, n, (int)xn, n, 1.0f, lhi, llo, w.bhi, w.blo, NB, 0.0f, Xi, d, false,
                                     w.status, ss, xt));
            ss_k = true;
            if (m > 0 && !sp_last) {
                // B[k0+n : sp_end, 0:ncols] -= L21[0 : sp_end-k0-n] X_k
                GPTQ_CUDA_TRY(side_gemm((int)(sp_end - k0 - n), (int)ncols, n, Lhi, Llo, w.xhi + NB * j,
                                        w.xlo + NB * j, w.Binv + (k0 + n) * d, false));
            }
            if (m > 0 && sp_last) {
                // deferred: B[sp_end:, 0:sp_end] -= L[sp_end:, sp0:sp_end] X[sp0:sp_end, 0:sp_end]
                GPTQ_CUDA_TRY(side_gemm((int)(d - sp_end), (int)sp_end, (int)SPW, Ehi, Elo, w.xhi, w.xlo,
                                        w.Binv + sp_end * d, false));
            }
            GPTQ_CUDA_TRY(record(two ? conc->side_done[par] : nullptr, ss));
            if (sp_last) GPTQ_CUDA_TRY(record(two ? conc->far_done[spar] : nullptr, ss));
        }
        if (two) {
            GPTQ_CUDA_TRY(record(conc->join_side, ss));
            GPTQ_CUDA_TRY(record(conc->join_crit, cs));
            GPTQ_CUDA_TRY(wait(s, conc->join_side));
            GPTQ_CUDA_TRY(wait(s, conc->join_crit));
        }
    } else {
        // blocked right-looking Cholesky of A (lower), FFMA trailing products
        for (int64_t kb = 0; kb < nblk; ++kb) {
            const int64_t k0 = kb * NB;
            const int n = (int)std::min<int64_t>(NB, d - k0);
            float* LinvK = w.LinvD + kb * NB * NB;
            GPTQ_LAUNCH(K_POTRF, s, potrf_diag_kernel<<<1, 512, potrf_smem, s>>>(w.A, d, k0, n, LinvK, nullptr,
                                                                                 nullptr, 1, w.status));
            GPTQ_LAUNCH_CHECK();
            const int64_t m = d - k0 - n;
            if (m <= 0) continue;
            float* P = w.A + (k0 + n) * d + k0;
            GPTQ_CUDA_TRY(sgemm(K_SGEMM_PREP, true, (int)m, n, n, 1.0f, P, d, LinvK, NB, 0.0f, P, d, false, s));
            GPTQ_CUDA_TRY(sgemm(K_SGEMM_PREP, true, (int)m, (int)m, n, -1.0f, P, d, P, d, 1.0f,
                                w.A + (k0 + n) * d + k0 + n, d, true, s));
        }
        // L^-1 by block rows: X[i,:] = Linv_ii * B[i,:];  B[i+1:, :] -= L[i+1:, i] X[i, :]
        for (int64_t ib = 0; ib < nblk; ++ib) {
            const int64_t i0 = ib * NB;
            const int n = (int)std::min<int64_t>(NB, d - i0);
            const int64_t ncols = i0 + n;
            float* Xi = w.Binv + i0 * d;
            const int64_t m = d - i0 - n;
            GPTQ_CUDA_TRY(sgemm(K_SGEMM_PREP, false, n, (int)ncols, n, 1.0f, w.LinvD + ib * NB * NB, NB, Xi, d, 0.0f,
                                Xi, d, false, s));
            if (m > 0)
                GPTQ_CUDA_TRY(sgemm(K_SGEMM_PREP, false, (int)m, (int)ncols, n, -1.0f, w.A + (i0 + n) * d + i0, d, Xi,
                                    d, 1.0f, w.Binv + (i0 + n) * d, d, false, s));
        }
    }

    if (vec4) {
        GPTQ_LAUNCH(K_SCATTER, s, prep_scatter4_kernel<<<(unsigned)ceil_div(d, SCR_ROWS), 256, 0, s>>>(w.Binv, d, perm,
                                                                                                       w.rr, U));
        GPTQ_LAUNCH_CHECK();
    } else {
        dim3 grid((unsigned)std::min<int64_t>(ceil_div(d, 256), 64), (unsigned)d);
        GPTQ_LAUNCH(K_SCATTER, s, prep_scatter_kernel<<<grid, 256, 0, s>>>(w.Binv, d, perm, w.rr, U));
        GPTQ_LAUNCH_CHECK();
    }

    return finish_call(w.status, s);
}

}  // namespace
}  // namespace gptq

extern "C" int gptq_prepare(const float* H, const float* diag_xtx, int64_t d, float damp, int act_order, float* U,
                            int32_t* perm, uint8_t* dead, void* ws, size_t ws_bytes, void* stream) {
    const int arg = check_args(H, diag_xtx, d, damp, act_order, U, perm, dead, ws, ws_bytes);
    if (arg != GPTQ_OK) return arg;
    int dev = 0;
    GPTQ_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kMaxPrepDevices || d <= NB)
        return prepare_impl(H, diag_xtx, d, damp, act_order, U, perm, dead, ws, ws_bytes, stream, nullptr);
    PrepConcurrency& c = conc_for(dev, static_cast<cudaStream_t>(stream));
    std::lock_guard<std::mutex> lk(c.mu);
    if (conc_init(c, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        (void)cudaGetLastError();
        return GPTQ_ERR_CUDA;
    }
    return prepare_impl(H, diag_xtx, d, damp, act_order, U, perm, dead, ws, ws_bytes, stream, &c);
}

// ------------------------------------------------------------------------------------
// gptq_prepare_noalloc: gptq_prepare for callers that cannot allocate device memory.
//
// Some callers of this library cannot call cudaMalloc for the workspace: a host
// framework that owns every byte of device memory through its own pool and hands out
// nothing extra, or a latency-sensitive path that cannot take cudaMalloc's implicit
// device synchronisation. For them this entry point uses a fixed scratch area compiled
// into the library as a file-scope __device__ array, sized for d <= kNoAllocMaxD.
// Every GPU that loads the library holds this array (about 14 MiB) until the process
// exits. The entry point itself allocates nothing: no cudaMalloc, cudaFree or allocating
// library routine.
// ------------------------------------------------------------------------------------
namespace gptq {
namespace {

constexpr int64_t kNoAllocMaxD = 1024;

// the workspace gptq_prepare carves for d = kNoAllocMaxD
constexpr size_t kNoAllocBytes = prep_ws_bytes(kNoAllocMaxD);

// Host code must not use this name as an address: on the host it is only a stand-in for
// the device symbol. The device address comes from cudaGetSymbolAddress, per CUDA context.
static __device__ __align__(256) unsigned char g_prepare_scratch[kNoAllocBytes];

// the array's address in each CUDA context that has called the entry point (keyed by the
// context's unique id: a device reset or another context on the same device gets its own
// lookup, never a stale address)
ContextPtrCache g_noalloc_addr;

}  // namespace
}  // namespace gptq

extern "C" int gptq_prepare_noalloc(const float* H, const float* diag_xtx, int64_t d, float damp, int act_order,
                                    float* U, int32_t* perm, uint8_t* dead, void* stream) {
    using namespace gptq;
    if (d <= 0) return GPTQ_ERR_INVALID_ARG;
    if (d > kNoAllocMaxD) return GPTQ_ERR_UNSUPPORTED;
    const size_t need = gptq_prepare_workspace_bytes(d, act_order);
    if (need > kNoAllocBytes) return GPTQ_ERR_UNSUPPORTED;
    void* scratch = g_noalloc_addr.find(current_context_id());
    if (!scratch) {
        // first call in this context: look up this context's copy of the array (once)
        const cudaError_t e = cudaGetSymbolAddress(&scratch, g_prepare_scratch);
        if (e != cudaSuccess || scratch == nullptr) {
            (void)cudaGetLastError();
            return GPTQ_ERR_CUDA;
        }
        g_noalloc_addr.put(current_context_id(), scratch);   // the lookup made the context current
    }
    // every slab gptq_prepare reads is written by it first (its status word is cleared),
    // so the previous call's contents need no clearing here
    // one stream: no streams or events are created for this entry point
    return prepare_impl(H, diag_xtx, d, damp, act_order, U, perm, dead, scratch, kNoAllocBytes, stream, nullptr);
}
