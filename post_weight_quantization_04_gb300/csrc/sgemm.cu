// sgemm.cu — fp32 FFMA tiled GEMM: C = beta * C + alpha * A * op(B).
//
// Used where the path needs fp32-accurate contractions: the trailing updates of the
// blocked Cholesky factorisation and triangular inverse, and GPTQ's lazy trailing update
// W[:, e:] -= Err * U[blk, e:].
//
// Tiling: 128x128 C tile per 256-thread CTA, 8x8 outputs per thread (two 4x4 sub-tiles
// per dimension so shared-memory reads are broadcast / conflict free), K in steps of 8
// double-buffered through shared memory. Bounds are checked on every global access, so
// any M, N, K, leading dimension and alignment is accepted.
//
// Aliasing: C may alias A when N <= 128 (each CTA then owns whole rows of C and reads all
// of its rows of A before writing), or alias B when M <= 128 and op(B) = B (each CTA owns
// whole columns). Callers rely on this for in-place triangular multiplies.
#include "common.cuh"
#include "sgemm.cuh"

namespace gptq {

namespace {

constexpr int BM = 128, BN = 128, BK = 8, PAD = 4, NT = 256;

template <bool TRANS_B>
__global__ void __launch_bounds__(NT) sgemm_kernel(int M, int N, int K, float alpha, const float* A, int64_t lda,
                                                  const float* B, int64_t ldb, float beta, float* C, int64_t ldc,
                                                  int lower_only) {
    const int m0 = blockIdx.y * BM;
    const int n0 = blockIdx.x * BN;
    if (lower_only && n0 > m0 + BM - 1) return;  // tile entirely above the diagonal

    __shared__ __align__(16) float As[2][BK][BM + PAD];
    __shared__ __align__(16) float Bs[2][BK][BN + PAD];

    const int tid = threadIdx.x;
    const int tx = tid & 15, ty = tid >> 4;

    // global -> register staging
    // A tile (BM x BK): thread loads row ar, k columns ak..ak+3
    const int ar = tid >> 1, ak = (tid & 1) * 4;
    // B tile: !TRANS_B: (BK x BN) row bk, cols bn..bn+3 ; TRANS_B: row (n) bn_t, k bk_t..bk_t+3
    const int bk = tid >> 5, bn = (tid & 31) * 4;
    const int bn_t = tid >> 1, bk_t = (tid & 1) * 4;

    float ra[4], rb[4];
    auto load_tile = [&](int k0) {
        const int gm = m0 + ar;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int gk = k0 + ak + i;
            ra[i] = (gm < M && gk < K) ? A[(int64_t)gm * lda + gk] : 0.0f;
        }
        if (!TRANS_B) {
            const int gk = k0 + bk;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int gn = n0 + bn + i;
                rb[i] = (gk < K && gn < N) ? B[(int64_t)gk * ldb + gn] : 0.0f;
            }
        } else {
            const int gn = n0 + bn_t;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int gk = k0 + bk_t + i;
                rb[i] = (gk < K && gn < N) ? B[(int64_t)gn * ldb + gk] : 0.0f;
            }
        }
    };
    auto store_tile = [&](int buf) {
#pragma unroll
        for (int i = 0; i < 4; ++i) As[buf][ak + i][ar] = ra[i];
        if (!TRANS_B) {
            *reinterpret_cast<float4*>(&Bs[buf][bk][bn]) = make_float4(rb[0], rb[1], rb[2], rb[3]);
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) Bs[buf][bk_t + i][bn_t] = rb[i];
        }
    };

    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;

    const int ktiles = (K + BK - 1) / BK;
    load_tile(0);
    store_tile(0);
    __syncthreads();
    for (int kt = 0; kt < ktiles; ++kt) {
        const int buf = kt & 1;
        if (kt + 1 < ktiles) load_tile((kt + 1) * BK);
#pragma unroll
        for (int k = 0; k < BK; ++k) {
            float a[8], b[8];
            const float4 a0 = *reinterpret_cast<const float4*>(&As[buf][k][ty * 4]);
            const float4 a1 = *reinterpret_cast<const float4*>(&As[buf][k][64 + ty * 4]);
            const float4 b0 = *reinterpret_cast<const float4*>(&Bs[buf][k][tx * 4]);
            const float4 b1 = *reinterpret_cast<const float4*>(&Bs[buf][k][64 + tx * 4]);
            a[0] = a0.x; a[1] = a0.y; a[2] = a0.z; a[3] = a0.w;
            a[4] = a1.x; a[5] = a1.y; a[6] = a1.z; a[7] = a1.w;
            b[0] = b0.x; b[1] = b0.y; b[2] = b0.z; b[3] = b0.w;
            b[4] = b1.x; b[5] = b1.y; b[6] = b1.z; b[7] = b1.w;
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        if (kt + 1 < ktiles) store_tile(buf ^ 1);
        __syncthreads();
    }

#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int gm = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
        if (gm >= M) continue;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int gn = n0 + (j < 4 ? tx * 4 + j : 64 + tx * 4 + (j - 4));
            if (gn >= N) continue;
            float* c = C + (int64_t)gm * ldc + gn;
            const float v = alpha * acc[i][j];
            *c = (beta == 0.0f) ? v : fmaf(beta, *c, v);
        }
    }
}

}  // namespace

cudaError_t sgemm(int id, bool trans_b, int M, int N, int K, float alpha, const float* A, int64_t lda, const float* B,
                  int64_t ldb, float beta, float* C, int64_t ldc, bool lower_only, cudaStream_t stream) {
    if (M <= 0 || N <= 0) return cudaSuccess;
    dim3 grid((unsigned)((N + BN - 1) / BN), (unsigned)((M + BM - 1) / BM));
    if (trans_b)
        GPTQ_LAUNCH(id, stream, sgemm_kernel<true><<<grid, NT, 0, stream>>>(M, N, K, alpha, A, lda, B, ldb, beta, C,
                                                                            ldc, lower_only ? 1 : 0));
    else
        GPTQ_LAUNCH(id, stream, sgemm_kernel<false><<<grid, NT, 0, stream>>>(M, N, K, alpha, A, lda, B, ldb, beta, C,
                                                                             ldc, lower_only ? 1 : 0));
    return cudaGetLastError();
}

}  // namespace gptq
