// Launchers of the NVFP4 quantizer kernels.
#pragma once
#include "common.cuh"

namespace impfp4 {

// Number of SMs of the current device (cached per device).
int num_sms();

// Workspace (bytes) of launch_quantize for a rows x K tensor.
size_t quantize_workspace_bytes(int64_t rows, int64_t K);

// Enqueue the two quantizer passes on `stream`.  Arguments are validated by
// the caller (api.cu).  rows > 0.
cudaError_t launch_quantize(const uint16_t *x, int64_t rows, int64_t K, int64_t ldx,
                            uint8_t *codes, uint8_t *scales, float *tensor_scale,
                            int32_t *status, void *workspace, cudaStream_t stream);

}  // namespace impfp4
