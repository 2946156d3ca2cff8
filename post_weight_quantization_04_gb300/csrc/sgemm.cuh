// sgemm.cuh — host launcher of the fp32 FFMA tiled GEMM (see sgemm.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace gptq {

// C[M x N] = beta * C + alpha * A[M x K] * op(B); op(B) = B (K x N, row-major) or, with
// trans_b, B^T for B stored N x K row-major. lower_only skips C tiles that lie entirely
// above the diagonal (row < col everywhere in the tile).
cudaError_t sgemm(int id, bool trans_b, int M, int N, int K, float alpha, const float* A, int64_t lda, const float* B,
                  int64_t ldb, float beta, float* C, int64_t ldc, bool lower_only, cudaStream_t stream);

}  // namespace gptq
