// Launcher of the prefill GEMM on the block-scaled FP4 tensor cores.
#pragma once
#include "common.cuh"

namespace impfp4 {

int num_sms();

// Dynamic shared memory of the GEMM kernel (bytes).
size_t gemm_mxf4_smem_bytes();

// Workspace (bytes, on the current device) of the stream-K schedule:
// per-tile counters and one partial 128 x 256 fp32 tile per CTA and segment.
size_t gemm_mxf4_workspace_bytes(int64_t M, int64_t N, int64_t K);

// A launch of the GEMM with its tensor maps built and the kernel's
// shared-memory size set, so that enqueueing it cannot fail on either.
struct GemmMxf4Plan {
  struct Impl;
  Impl *impl;
  GemmMxf4Plan();
  ~GemmMxf4Plan();
  GemmMxf4Plan(const GemmMxf4Plan &) = delete;
  GemmMxf4Plan &operator=(const GemmMxf4Plan &) = delete;
};

// Plan Y[M][N] = s_x * s_w * (Xq . Wq^T) with both operands NVFP4: X codes
// row-major [M][K/2]; W codes row-major [N][K/2] or, with w_tiled, in the
// 16 KB tile layout (quantize.cuh); block scales of both in the tensor-core
// atom layout.  K % 64 == 0; arrays 16-byte aligned.  With a workspace
// (gemm_mxf4_workspace_bytes, 16-byte aligned) the (tile, K stage) work is
// split evenly over the CTAs (stream-K); without one each CTA takes whole
// tiles.  Enqueues nothing.
cudaError_t plan_gemm_mxf4(const uint8_t *x_codes, const uint8_t *x_mma_scales, const float *s_x,
                           const uint8_t *w_codes, bool w_tiled, const uint8_t *w_mma_scales,
                           const float *s_w, int64_t M, int64_t N, int64_t K, uint16_t *y,
                           int64_t ldy, int32_t *status, void *workspace, GemmMxf4Plan &plan);

// Plan the SwiGLU form: h[M][N] = silu(s_x s_g (Xq . Wg^T)) * s_x s_u (Xq . Wu^T),
// gate and up weights in the tile layout (same N and K), whole tiles of 128
// output columns; the kernel folds max|h| (bf16 magnitude bits) into
// *h_amax with atomicMax (the caller zeroes it).  Enqueues nothing.
cudaError_t plan_gemm_mxf4_swiglu(const uint8_t *x_codes, const uint8_t *x_mma_scales,
                                  const float *s_x, const uint8_t *gate_tiles,
                                  const uint8_t *gate_scales, const float *s_gate,
                                  const uint8_t *up_tiles, const uint8_t *up_scales,
                                  const float *s_up, int64_t M, int64_t N, int64_t K, uint16_t *h,
                                  int64_t ldh, uint32_t *h_amax, int32_t *status,
                                  GemmMxf4Plan &plan);

// Enqueue a planned GEMM on `stream`.
cudaError_t enqueue_gemm_mxf4(const GemmMxf4Plan &plan, cudaStream_t stream);

}  // namespace impfp4
