// Launchers of the NVFP4 quantizer kernels.
#pragma once
#include "common.cuh"

namespace impfp4 {

// Number of SMs of the current device (cached per device).
int num_sms();

// Workspace (bytes) of launch_quantize for a rows x K tensor.
size_t quantize_workspace_bytes(int64_t rows, int64_t K);

// Bytes of the fixed scratch array of the allocation-free quantizer.
size_t quantize_noalloc_capacity();

// The two quantizer passes with their scratch in a fixed device array (no
// caller workspace, no allocation).  Calls that overlap on the GPU share the
// array and race.
cudaError_t launch_quantize_noalloc(const uint16_t *x, int64_t rows, int64_t K, int64_t ldx,
                                    uint8_t *codes, uint8_t *scales, float *tensor_scale,
                                    int32_t *status, cudaStream_t stream);

// MXFP4 quantizer (one pass, no workspace): codes [rows][K/2], E8M0 scales
// [rows][K/32].  K % 32 == 0.
cudaError_t launch_mx_quantize(const uint16_t *x, int64_t rows, int64_t K, int64_t ldx,
                               uint8_t *codes, uint8_t *scales, int32_t *status,
                               cudaStream_t stream);

// FP8-E4M3 weight quantizer: the global amax pass (workspace as for
// launch_quantize), then codes [rows][K] and s8 = g / 448.  K % 16 == 0.
cudaError_t launch_fp8_quantize(const uint16_t *x, int64_t rows, int64_t K, int64_t ldx,
                                uint8_t *codes, float *tensor_scale, int32_t *status,
                                void *workspace, cudaStream_t stream);

// MXFP4 -> the same values in NVFP4 form (codes copied unless out_codes ==
// codes; E4M3 half-block scales; power-of-two tensor scale).  workspace: 4
// bytes, 4-byte aligned.
cudaError_t launch_mx_to_nvfp4(const uint8_t *codes, const uint8_t *mx_scales, int64_t rows,
                               int64_t K, uint8_t *out_codes, uint8_t *nv_scales,
                               float *tensor_scale, int32_t *status, void *workspace,
                               cudaStream_t stream);

// Enqueue the two quantizer passes on `stream`.  Arguments are validated by
// the caller (api.cu).  rows > 0.
cudaError_t launch_quantize(const uint16_t *x, int64_t rows, int64_t K, int64_t ldx,
                            uint8_t *codes, uint8_t *scales, float *tensor_scale,
                            int32_t *status, void *workspace, cudaStream_t stream);

}  // namespace impfp4

namespace impfp4 {

// ---- block-scale layout used by the tensor-core (prefill) path -------------
//
// tcgen05.cp (shape 32x128b, warpx4) moves 512-byte scale "atoms" into tensor
// memory; one atom holds the scales of 128 rows x 4 blocks (64 k), row r of
// the atom at byte 16*(r % 32) + 4*((r / 32) % 4), block kb at + kb.  In
// global memory the atoms of a 128-row block are stored consecutively along
// K, and row blocks follow each other.  Rows are padded to a multiple of 256
// so a 256-row operand tile never reads past the array.
__host__ __device__ inline int64_t mma_scale_rows(int64_t rows) { return ((rows + 255) / 256) * 256; }
__host__ __device__ inline size_t mma_scale_bytes(int64_t rows, int64_t K) {
  return (size_t)mma_scale_rows(rows) * (size_t)(K / 16);
}
__host__ __device__ inline int64_t mma_scale_offset(int64_t r, int64_t kb, int64_t K) {
  const int64_t atoms_per_rowblock = K / 64;
  return ((r / 128) * atoms_per_rowblock + kb / 4) * 512 + 16 * (r % 32) + 4 * ((r / 32) % 4) +
         (kb % 4);
}

// ---- code layout used by the tensor-core paths --------------------------------
//
// The E2M1 codes of a weight in "tiles": 128 rows x 256 elements (128 bytes
// per row, 16 KB per tile), each tile stored exactly as a 128-byte-swizzled
// shared-memory operand tile (row rr at rr * 128, its 16-byte unit u at unit
// u ^ (rr % 8)), so one contiguous copy of 16 KB loads it.  Tiles run along K
// (K padded to a multiple of 256), then down the rows (rows padded to a
// multiple of 256, like the scales).  Padding is zero.
__host__ __device__ inline int64_t mma_code_chunks(int64_t K) { return (K + 255) / 256; }
__host__ __device__ inline size_t mma_code_bytes(int64_t rows, int64_t K) {
  return (size_t)mma_scale_rows(rows) * (size_t)mma_code_chunks(K) * 128;
}
// Byte offset of the tile (row block rb of 128 rows, K chunk c of 256).
__host__ __device__ inline int64_t mma_code_tile(int64_t rb, int64_t c, int64_t K) {
  return (rb * mma_code_chunks(K) + c) * 16384;
}

// Row-major codes [rows][K/2] -> the tile layout above.
cudaError_t launch_code_relayout(const uint8_t *codes, int64_t rows, int64_t K, uint8_t *mma_codes,
                                 cudaStream_t stream);

// Row-major scales [rows][K/16] -> the atom layout above (padding rows = 0).
cudaError_t launch_scale_relayout(const uint8_t *scales, int64_t rows, int64_t K,
                                  uint8_t *mma_scales, cudaStream_t stream);

// The encode pass alone, the global amax given (bf16 magnitude bits of
// max|x| in device memory, e.g. folded by the SwiGLU GEMM epilogue);
// scales row-major or (mma_layout) in the atom layout.
cudaError_t launch_encode_with_amax(const uint16_t *x, int64_t rows, int64_t K, int64_t ldx,
                                   const uint32_t *amax_bits, uint8_t *codes, uint8_t *scales,
                                   float *tensor_scale, bool mma_layout, cudaStream_t stream);

// The quantizer writing its block scales in the atom layout (codes stay
// row-major [rows][K/2]).  K % 64 == 0.
cudaError_t launch_quantize_mma(const uint16_t *x, int64_t rows, int64_t K, int64_t ldx,
                                uint8_t *codes, uint8_t *mma_scales, float *tensor_scale,
                                int32_t *status, void *workspace, cudaStream_t stream);

}  // namespace impfp4
