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

constexpr int BK = 8, PAD = 4, NT = 256;

// BM x BN tile per 256-thread CTA (16 x 16 threads); each thread owns TM x TN outputs
// as two row halves and two column halves (TM/2 and TN/2 contiguous), so the shared-
// memory reads of a warp are broadcasts or conflict free.
template <int BM, int BN, bool TRANS_B>
__global__ void __launch_bounds__(NT) sgemm_kernel(int M, int N, int K, float alpha, const float* A, int64_t lda,
                                                  const float* B, int64_t ldb, float beta, float* C, int64_t ldc,
                                                  int lower_only) {
    constexpr int TM = BM / 16, TN = BN / 16, HM = TM / 2, HN = TN / 2;
    constexpr int LA = BM * BK / NT, LB = BN * BK / NT;  // elements per thread per tile load
    const int m0 = blockIdx.y * BM;
    const int n0 = blockIdx.x * BN;
    if (lower_only && n0 > m0 + BM - 1) return;  // tile entirely above the diagonal

    __shared__ __align__(16) float As[2][BK][BM + PAD];
    __shared__ __align__(16) float Bs[2][BK][BN + PAD];

    const int tid = threadIdx.x;
    const int tx = tid & 15, ty = tid >> 4;
    const int ar = tid / (BK / LA), ak = (tid % (BK / LA)) * LA;
    const int bk = tid / (BN / LB), bn = (tid % (BN / LB)) * LB;
    const int bn_t = tid / (BK / LB), bk_t = (tid % (BK / LB)) * LB;

    float ra[LA], rb[LB];
    auto load_tile = [&](int k0) {
        const int gm = m0 + ar;
#pragma unroll
        for (int i = 0; i < LA; ++i) {
            const int gk = k0 + ak + i;
            ra[i] = (gm < M && gk < K) ? A[(int64_t)gm * lda + gk] : 0.0f;
        }
        if (!TRANS_B) {
            const int gk = k0 + bk;
#pragma unroll
            for (int i = 0; i < LB; ++i) {
                const int gn = n0 + bn + i;
                rb[i] = (gk < K && gn < N) ? B[(int64_t)gk * ldb + gn] : 0.0f;
            }
        } else {
            const int gn = n0 + bn_t;
#pragma unroll
            for (int i = 0; i < LB; ++i) {
                const int gk = k0 + bk_t + i;
                rb[i] = (gk < K && gn < N) ? B[(int64_t)gn * ldb + gk] : 0.0f;
            }
        }
    };
    auto store_tile = [&](int buf) {
#pragma unroll
        for (int i = 0; i < LA; ++i) As[buf][ak + i][ar] = ra[i];
        if (!TRANS_B) {
#pragma unroll
            for (int i = 0; i < LB; ++i) Bs[buf][bk][bn + i] = rb[i];
        } else {
#pragma unroll
            for (int i = 0; i < LB; ++i) Bs[buf][bk_t + i][bn_t] = rb[i];
        }
    };

    float acc[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = 0.0f;

    const int ktiles = (K + BK - 1) / BK;
    load_tile(0);
    store_tile(0);
    __syncthreads();
    for (int kt = 0; kt < ktiles; ++kt) {
        const int buf = kt & 1;
        if (kt + 1 < ktiles) load_tile((kt + 1) * BK);
#pragma unroll
        for (int k = 0; k < BK; ++k) {
            float a[TM], b[TN];
#pragma unroll
            for (int i = 0; i < HM; ++i) {
                a[i] = As[buf][k][ty * HM + i];
                a[HM + i] = As[buf][k][BM / 2 + ty * HM + i];
            }
#pragma unroll
            for (int j = 0; j < HN; ++j) {
                b[j] = Bs[buf][k][tx * HN + j];
                b[HN + j] = Bs[buf][k][BN / 2 + tx * HN + j];
            }
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        if (kt + 1 < ktiles) store_tile(buf ^ 1);
        __syncthreads();
    }

#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int gm = m0 + (i < HM ? ty * HM + i : BM / 2 + ty * HM + (i - HM));
        if (gm >= M) continue;
#pragma unroll
        for (int j = 0; j < TN; ++j) {
            const int gn = n0 + (j < HN ? tx * HN + j : BN / 2 + tx * HN + (j - HN));
            if (gn >= N) continue;
            float* c = C + (int64_t)gm * ldc + gn;
            const float v = alpha * acc[i][j];
            *c = (beta == 0.0f) ? v : fmaf(beta, *c, v);
        }
    }
}

template <int T>
void launch(int id, bool trans_b, int M, int N, int K, float alpha, const float* A, int64_t lda, const float* B,
            int64_t ldb, float beta, float* C, int64_t ldc, bool lower_only, cudaStream_t stream) {
    dim3 grid((unsigned)((N + T - 1) / T), (unsigned)((M + T - 1) / T));
    if (trans_b)
        GPTQ_LAUNCH(id, stream, sgemm_kernel<T, T, true><<<grid, NT, 0, stream>>>(M, N, K, alpha, A, lda, B, ldb,
                                                                                  beta, C, ldc, lower_only ? 1 : 0));
    else
        GPTQ_LAUNCH(id, stream, sgemm_kernel<T, T, false><<<grid, NT, 0, stream>>>(M, N, K, alpha, A, lda, B, ldb,
                                                                                   beta, C, ldc, lower_only ? 1 : 0));
}

}  // namespace

cudaError_t sgemm(int id, bool trans_b, int M, int N, int K, float alpha, const float* A, int64_t lda, const float* B,
                  int64_t ldb, float beta, float* C, int64_t ldc, bool lower_only, cudaStream_t stream) {
    if (M <= 0 || N <= 0) return cudaSuccess;
    // 64 x 64 tiles when 128 x 128 tiles would leave SMs idle; never for in-place calls,
    // whose safety needs one CTA to own whole rows (C == A) or whole columns (C == B)
    const bool aliased = (C == A) || (C == B);
    int64_t tiles = (int64_t)((M + 127) / 128) * ((N + 127) / 128);
    if (lower_only) tiles = (tiles + (M + 127) / 128) / 2;
    static const int sms = device_sm_count();
    if (!aliased && tiles < sms)
        launch<64>(id, trans_b, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, lower_only, stream);
    else
        launch<128>(id, trans_b, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, lower_only, stream);
    return cudaGetLastError();
}

}  // namespace gptq
