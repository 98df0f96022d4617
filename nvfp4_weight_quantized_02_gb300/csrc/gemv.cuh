// Launcher of the decode-path GEMV / skinny GEMM (M <= 16).
#pragma once
#include "common.cuh"

namespace impfp4 {

constexpr int64_t kDecodeMaxM = 16;

int num_sms();

// True if launch_gemv has a launch plan for this shape.
bool gemv_supported(int64_t M, int64_t N, int64_t K);

// Enqueue Y[M][N] = X[M][K] * W^T (bf16 X and Y, NVFP4 W) on `stream`.
// Arguments are validated by the caller.  1 <= M <= 16, N >= 1, K % 64 == 0.
cudaError_t launch_gemv(const uint16_t *x, int64_t M, int64_t K, int64_t ldx, const uint8_t *codes,
                        const uint8_t *scales, const float *tensor_scale, int64_t N, uint16_t *y,
                        int64_t ldy, int32_t *status, cudaStream_t stream);

// The tensor-core GEMV (gemv_tc.cu): passes of 1, 2, 4 or 8 rows of X,
// each one stream of W.
bool gemv_tc_supported(int64_t M, int64_t N, int64_t K);
cudaError_t launch_gemv_tc(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                           const uint8_t *codes, const uint8_t *scales, const float *tensor_scale,
                           int64_t N, uint16_t *y, int64_t ldy, int32_t *status,
                           cudaStream_t stream);

}  // namespace impfp4
