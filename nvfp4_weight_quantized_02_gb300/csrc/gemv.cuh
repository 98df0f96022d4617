// Launcher of the decode-path GEMV / skinny GEMM (M <= 16).
#pragma once
#include "common.cuh"

namespace impfp4 {

constexpr int64_t kDecodeMaxM = 16;

int num_sms();

// True if launch_gemv has a launch plan for this shape.
bool gemv_supported(int64_t M, int64_t N, int64_t K);

// Kernel launches of one launch_gemv call given a workspace and 16-byte
// aligned W arrays, with the name of the kernel that streams W in *kernel
// (0: no plan).
int gemv_launches(int64_t M, int64_t N, int64_t K, const char **kernel);

// Enqueue Y[M][N] = X[M][K] * W^T (bf16 X and Y, NVFP4 W) on `stream`.
// Arguments are validated by the caller.  1 <= M <= 16, N >= 1, K % 64 == 0.
// `workspace` (gemv_f4_workspace_bytes, 16-byte aligned) enables the FP4
// tensor-core path for the shapes gemv_f4_shape_ok accepts; nullptr selects
// the f16 tensor-core / CUDA-core paths.
cudaError_t launch_gemv(const uint16_t *x, int64_t M, int64_t K, int64_t ldx, const uint8_t *codes,
                        const uint8_t *scales, const float *tensor_scale, int64_t N, uint16_t *y,
                        int64_t ldy, int32_t *status, void *workspace, cudaStream_t stream);

// The tensor-core GEMV (gemv_tc.cu): passes of 1, 2, 4 or 8 rows of X,
// each one stream of W.
bool gemv_tc_supported(int64_t M, int64_t N, int64_t K);
int gemv_tc_launches(int64_t M, int64_t N, int64_t K);  // passes; 0: no plan
cudaError_t launch_gemv_tc(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                           const uint8_t *codes, const uint8_t *scales, const float *tensor_scale,
                           int64_t N, uint16_t *y, int64_t ldy, int32_t *status,
                           cudaStream_t stream);

// The block-scaled FP4 tensor-core GEMV (gemv_f4.cu): X split into NVFP4
// components per call (needs a workspace), W streamed straight into
// tcgen05.mma.kind::mxf4nvf4.  One pass over W for every M <= 16.
bool gemv_f4_shape_ok(int64_t M, int64_t N, int64_t K);
size_t gemv_f4_workspace_bytes(int64_t M, int64_t N, int64_t K);
bool gemv_f4_supported(int64_t M, int64_t N, int64_t K, const void *codes, const void *scales);
int gemv_f4_launches(int64_t M, int64_t N, int64_t K, const char **kernel);
// `prepared`: codes and scales in the tensor-core (MMA) layout of
// quantize.cuh (contiguous 16 KB code tiles and 2 KB scale-atom runs per
// stage) instead of row-major.  `x2` (optional, bf16[M][ldx2]): X is then
// bf16(silu(x) * x2), formed where the split kernel reads it.
cudaError_t launch_gemv_f4(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                           const uint8_t *codes, const uint8_t *scales, const float *tensor_scale,
                           int64_t N, uint16_t *y, int64_t ldy, int32_t *status, void *workspace,
                           cudaStream_t stream, bool prepared = false,
                           const uint16_t *x2 = nullptr, int64_t ldx2 = 0);
// Kernel launches of a call with the SwiGLU X (x2 given): always through a
// split kernel; 0 if the FP4 decode path does not take the shape.
int gemv_f4_swiglu_launches(int64_t M, int64_t N, int64_t K, const char **kernel);

// Grouped decode GEMV: one X times up to four weights of the same K in one
// launch pair (the weights' tiles follow each other in one schedule; each
// keeps its tensor scale and output), weights in the MMA layout.
struct GemvGroup {
  const uint8_t *codes, *scales;  // MMA layout
  const float *tensor_scale;
  uint16_t *y;                    // bf16[M][ldy]
  int64_t N, ldy;
};
// True if launch_gemv_f4_grouped takes these groups (1 <= M <= 2,
// K % 256 == 0, K >= 1024, 1..4 groups, 16-byte aligned arrays).
bool gemv_f4_grouped_ok(int64_t M, int64_t K, const GemvGroup *g, int n);
size_t gemv_f4_grouped_workspace_bytes(int64_t M, int64_t K, const int64_t *N, int n);
cudaError_t launch_gemv_f4_grouped(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                                   const GemvGroup *g, int n, int32_t *status, void *workspace,
                                   cudaStream_t stream);

// Chained decode calls in one persistent launch (one CTA per SM, launched
// cooperatively): link c multiplies its X by its groups' weights (MMA
// layout, K = K of the link); dep: X is link c - 1's first output, which the
// kernel waits for.  1 <= M <= 2, at most four links.
struct ChainLink {
  const GemvGroup *g;
  int n;
  const uint16_t *x;
  int64_t ldx, K;
  bool dep;
  const uint16_t *x2 = nullptr;  // X = bf16(silu(x) * x2) when set (dep links)
  int64_t ldx2 = 0;
};
bool gemv_f4_chain_ok(int64_t M, const ChainLink *l, int n);
size_t gemv_f4_chain_workspace_bytes(int64_t M, const ChainLink *l, int n);
cudaError_t launch_gemv_f4_chain(int64_t M, const ChainLink *l, int n, int32_t *status,
                                 void *workspace, cudaStream_t stream);

// FP8-E4M3 weights (codes [N][K], one fp32 tensor scale): X split into E4M3
// components per call, W streamed into tcgen05.mma.kind::f8f6f4; passes of
// two rows of X.  K % 128 == 0, K >= 512, N >= 128.
bool gemv_fp8_shape_ok(int64_t M, int64_t N, int64_t K);
size_t gemv_fp8_workspace_bytes(int64_t N, int64_t K);
int gemv_fp8_launches(int64_t M);
cudaError_t launch_gemv_fp8(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                            const uint8_t *codes, const float *tensor_scale, int64_t N,
                            uint16_t *y, int64_t ldy, int32_t *status, void *workspace,
                            cudaStream_t stream);

}  // namespace impfp4
