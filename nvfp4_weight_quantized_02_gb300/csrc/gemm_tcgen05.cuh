// Launcher of the prefill GEMM on the block-scaled FP4 tensor cores.
#pragma once
#include "common.cuh"

namespace impfp4 {

int num_sms();

// Dynamic shared memory of the GEMM kernel (bytes).
size_t gemm_mxf4_smem_bytes();

// Y[M][N] = s_x * s_w * (Xq . Wq^T) with both operands NVFP4: X codes
// row-major [M][K/2]; W codes row-major [N][K/2] or, with w_tiled, in the
// 16 KB tile layout (quantize.cuh); block scales of both in the tensor-core
// atom layout.  K % 64 == 0; arrays 16-byte aligned.
cudaError_t launch_gemm_mxf4(const uint8_t *x_codes, const uint8_t *x_mma_scales,
                             const float *s_x, const uint8_t *w_codes, bool w_tiled,
                             const uint8_t *w_mma_scales, const float *s_w, int64_t M,
                             int64_t N, int64_t K, uint16_t *y, int64_t ldy, int32_t *status,
                             cudaStream_t stream);

}  // namespace impfp4
