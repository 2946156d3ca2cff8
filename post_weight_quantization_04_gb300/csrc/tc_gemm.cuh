// tc_gemm.cuh — fp32-accurate NT GEMM on the tensor cores (3xTF32), and the operand splits.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gptq {

// cuTensorMapEncodeTiled from the driver (looked up once), or null if unavailable.
PFN_cuTensorMapEncodeTiled_v12000 tma_encoder();

// A (rows x K, row stride lda) -> hi, lo (rows x ldk, dense), hi = A with the low 13
// mantissa bits cleared (exactly representable in TF32), lo = A - hi (exact in fp32).
// Columns K..ldk-1 of hi/lo are left untouched (the GEMM never reads them).
// pdl: launch as a programmatic dependent of the previous kernel in the stream (the
// kernels wait for it before touching global memory).
cudaError_t split_rows(int id, const float* A, int64_t lda, int rows, int K, float* hi, float* lo, int ldk,
                       cudaStream_t s, bool pdl = false);

// The same for the transpose of a (K x N, row stride ld) block: hi/lo are (N x ldk) with
// hi[n][k] = split(B[k][n]). strict_lower: only the entries n > k are needed (the reader
// takes hi/lo strictly below the diagonal only), so 64 x 64 tiles with every n < k are
// skipped and left unwritten.
cudaError_t split_cols(int id, const float* B, int64_t ld, int K, int N, float* hi, float* lo, int ldk,
                       cudaStream_t s, bool pdl = false, bool strict_lower = false);

// C[M x N] (ldc) = beta * C + alpha * (A * B^T) with A given as (Ahi, Alo) M x K and B as
// (Bhi, Blo) N x K, both K-major with row stride ldk (ldk % 4 == 0, 16-byte aligned).
// Products Ahi*Bhi + Ahi*Blo + Alo*Bhi on tcgen05 (kind::tf32), fp32 accumulation in TMEM.
// lower_only skips 128 x 128 C tiles entirely above the diagonal. C must not overlap the
// operands. Returns false (nothing launched) if C's stride or alignment rules out the
// vectorised epilogue; the caller then uses the FFMA path.
// Extra options: ldb, the row stride of Bhi/Blo (0 = same as ldk, the stride of Ahi/Alo);
// an optional TF32 split of the result, written by the epilogue: mode 1 hi[r][c], mode 2
// (transposed) hi[c][r], with row stride ld; max_ctas, a cap on the persistent grid
// (0 = one CTA per SM) that leaves SMs free for work on another stream; and pdl, launch
// as a programmatic dependent of the previous kernel in the stream (set up shared
// memory and TMEM while it finishes); row0, the first row of C the split output covers;
// narrow_ok, a latency-critical launch that may use 128 x 64 tiles (twice the CTAs, each
// with half the epilogue) when those still fit in one wave.
struct GemmOpts {
    float* hi = nullptr;
    float* lo = nullptr;
    int64_t ld = 0;
    int mode = 0;
    int64_t ldb = 0;
    int max_ctas = 0;
    bool pdl = false;
    int64_t row0 = 0;   // the split output covers rows >= row0 of C, stored from row 0
    bool narrow_ok = false;   // latency-critical: 64-column tiles allowed when they fit one wave
};
bool tc_gemm_nt_ok(const float* C, int64_t ldc);
cudaError_t tc_gemm_nt(int id, int M, int N, int K, float alpha, const float* Ahi, const float* Alo, const float* Bhi,
                       const float* Blo, int ldk, float beta, float* C, int64_t ldc, bool lower_only, int* status,
                       cudaStream_t s, GemmOpts out = GemmOpts());

}  // namespace gptq
