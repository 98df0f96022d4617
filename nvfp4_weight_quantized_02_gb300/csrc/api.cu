// The C ABI of imp_nvfp4.h: argument validation, workspace sizing and
// dispatch to the quantizer, the decode path (M <= 16) and the prefill path.
#include "gemv.cuh"
#include "quantize.cuh"

namespace {

using impfp4::kDecodeMaxM;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

imp_status check_tensor(const imp_nvfp4_tensor *t, int64_t rows, int64_t K) {
  if (!t || !t->codes || !t->scales || !t->tensor_scale) return IMP_ERR_INVALID_ARG;
  if (t->rows != rows || t->K != K) return IMP_ERR_INVALID_ARG;
  if (!aligned16(t->codes) || !aligned16(t->scales) || !aligned4(t->tensor_scale))
    return IMP_ERR_MISALIGNED;
  return IMP_OK;
}

imp_status from_cuda(cudaError_t e) { return e == cudaSuccess ? IMP_OK : IMP_ERR_CUDA; }

}  // namespace

extern "C" {

const char *imp_status_string(imp_status status) {
  switch (status) {
    case IMP_OK: return "IMP_OK";
    case IMP_ERR_INVALID_ARG: return "IMP_ERR_INVALID_ARG";
    case IMP_ERR_UNSUPPORTED_SHAPE: return "IMP_ERR_UNSUPPORTED_SHAPE";
    case IMP_ERR_MISALIGNED: return "IMP_ERR_MISALIGNED";
    case IMP_ERR_WORKSPACE_TOO_SMALL: return "IMP_ERR_WORKSPACE_TOO_SMALL";
    case IMP_ERR_CUDA: return "IMP_ERR_CUDA";
  }
  return "IMP_ERR_UNKNOWN";
}

size_t imp_nvfp4_quantize_workspace_size(int64_t rows, int64_t K) {
  if (rows <= 0 || K <= 0) return 0;
  return impfp4::quantize_workspace_bytes(rows, K);
}

imp_status imp_nvfp4_quantize(const void *x_bf16, int64_t rows, int64_t K, int64_t ldx,
                              const imp_nvfp4_tensor *out, int32_t *dev_status, void *workspace,
                              size_t ws_bytes, void *stream) {
  if (rows < 0 || K <= 0) return rows < 0 ? IMP_ERR_INVALID_ARG : IMP_ERR_UNSUPPORTED_SHAPE;
  if (K % 16) return IMP_ERR_UNSUPPORTED_SHAPE;
  if (ldx < K) return IMP_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (rows == 0) {
    // Empty tensor: only the tensor scale (0) is written; codes and scales
    // may be NULL.
    if (!out || out->rows != 0 || out->K != K || !out->tensor_scale) return IMP_ERR_INVALID_ARG;
    if (!aligned4(out->tensor_scale)) return IMP_ERR_MISALIGNED;
    return from_cuda(cudaMemsetAsync(out->tensor_scale, 0, sizeof(float), s));
  }
  imp_status st = check_tensor(out, rows, K);
  if (st != IMP_OK) return st;
  if (!x_bf16) return IMP_ERR_INVALID_ARG;
  if (!aligned16(x_bf16) || ldx % 8) return IMP_ERR_MISALIGNED;
  const size_t need = impfp4::quantize_workspace_bytes(rows, K);
  if (!workspace || ws_bytes < need) return IMP_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned16(workspace)) return IMP_ERR_MISALIGNED;
  return from_cuda(impfp4::launch_quantize(static_cast<const uint16_t *>(x_bf16), rows, K, ldx,
                                           out->codes, out->scales, out->tensor_scale, dev_status,
                                           workspace, s));
}

size_t imp_nvfp4_gemm_workspace_size(int64_t M, int64_t N, int64_t K) {
  if (M <= 0 || N <= 0 || K <= 0) return 0;
  if (M <= kDecodeMaxM) return 0;
  return 0;
}

imp_status imp_nvfp4_gemm(const void *x_bf16, int64_t M, int64_t K, int64_t ldx,
                          const imp_nvfp4_tensor *w, void *y_bf16, int64_t ldy,
                          int32_t *dev_status, void *workspace, size_t ws_bytes, void *stream) {
  if (M < 0 || !w) return IMP_ERR_INVALID_ARG;
  if (K <= 0 || K % 64) return IMP_ERR_UNSUPPORTED_SHAPE;
  const int64_t N = w->rows;
  if (N < 0 || w->K != K) return IMP_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return IMP_OK;  // nothing to read or write
  imp_status st = check_tensor(w, N, K);
  if (st != IMP_OK) return st;
  if (!x_bf16 || !y_bf16) return IMP_ERR_INVALID_ARG;
  if (ldx < K || ldy < N) return IMP_ERR_INVALID_ARG;
  if (!aligned16(x_bf16) || !aligned16(y_bf16) || ldx % 8 || ldy % 8) return IMP_ERR_MISALIGNED;
  const size_t need = imp_nvfp4_gemm_workspace_size(M, N, K);
  if (need && (!workspace || ws_bytes < need)) return IMP_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (M <= kDecodeMaxM) {
    if (!impfp4::gemv_supported(M, N, K)) return IMP_ERR_UNSUPPORTED_SHAPE;
    return from_cuda(impfp4::launch_gemv(static_cast<const uint16_t *>(x_bf16), M, K, ldx,
                                         w->codes, w->scales, w->tensor_scale, N,
                                         static_cast<uint16_t *>(y_bf16), ldy, dev_status, s));
  }
  return IMP_ERR_UNSUPPORTED_SHAPE;
}

}  // extern "C"
