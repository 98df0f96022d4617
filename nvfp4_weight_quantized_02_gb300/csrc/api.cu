// The C ABI of imp_nvfp4.h: argument validation, workspace sizing and
// dispatch to the quantizer, the decode path (M <= 16) and the prefill path.
#include "gemm_tcgen05.cuh"
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

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

struct PrefillWs {
  size_t partial, xcodes, xsc, wsc, sx, total;
};
// Workspace of the prefill path: amax partials | X codes | X atom scales |
// W atom scales | s_x.  The GEMM runs whole tiles per CTA (its stream-K
// schedule, measured slower on the prefill shapes, is opt-in through
// imp_nvfp4_gemm_fp4).
PrefillWs prefill_ws(int64_t M, int64_t N, int64_t K) {
  PrefillWs w;
  w.partial = 0;
  w.xcodes = align256(impfp4::quantize_workspace_bytes(M, K));
  w.xsc = align256(w.xcodes + (size_t)M * (size_t)(K / 2));
  w.wsc = align256(w.xsc + impfp4::mma_scale_bytes(M, K));
  w.sx = align256(w.wsc + impfp4::mma_scale_bytes(N, K));
  w.total = w.sx + 256;
  return w;
}

// One thread waits, with the library's bounded wait, on an mbarrier that
// nothing ever arrives at: after the wait limit it reports IMP_DEV_TIMEOUT
// and returns, leaving the context usable.
__global__ void bounded_wait_selftest_kernel(int32_t *status) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  impfp4::mbar_init(&bar, 1);
  impfp4::fence_mbar_init();
  impfp4::mbar_wait_bounded(&bar, 0u, status);
}

}  // namespace

extern "C" {

imp_status imp_selftest_bounded_wait(int32_t *dev_status, void *stream) {
  if (!dev_status || !aligned4(dev_status)) return IMP_ERR_INVALID_ARG;
  bounded_wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(dev_status);
  return from_cuda(cudaGetLastError());
}

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

imp_status imp_nvfp4_quantize_noalloc(const void *x_bf16, int64_t rows, int64_t K, int64_t ldx,
                                      const imp_nvfp4_tensor *out, int32_t *dev_status,
                                      void *stream) {
  if (rows < 0 || K <= 0) return rows < 0 ? IMP_ERR_INVALID_ARG : IMP_ERR_UNSUPPORTED_SHAPE;
  if (K % 16) return IMP_ERR_UNSUPPORTED_SHAPE;
  if (ldx < K) return IMP_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (rows == 0) {
    if (!out || out->rows != 0 || out->K != K || !out->tensor_scale) return IMP_ERR_INVALID_ARG;
    if (!aligned4(out->tensor_scale)) return IMP_ERR_MISALIGNED;
    return from_cuda(cudaMemsetAsync(out->tensor_scale, 0, sizeof(float), s));
  }
  imp_status st = check_tensor(out, rows, K);
  if (st != IMP_OK) return st;
  if (!x_bf16) return IMP_ERR_INVALID_ARG;
  if (!aligned16(x_bf16) || ldx % 8) return IMP_ERR_MISALIGNED;
  // the built-in scratch must hold this call's partial maxima
  if (impfp4::quantize_workspace_bytes(rows, K) > impfp4::quantize_noalloc_capacity())
    return IMP_ERR_WORKSPACE_TOO_SMALL;
  return from_cuda(impfp4::launch_quantize_noalloc(static_cast<const uint16_t *>(x_bf16), rows,
                                                   K, ldx, out->codes, out->scales,
                                                   out->tensor_scale, dev_status, s));
}

size_t imp_nvfp4_gemm_workspace_size(int64_t M, int64_t N, int64_t K) {
  if (M <= 0 || N <= 0 || K <= 0 || K % 64) return 0;
  if (M <= kDecodeMaxM)
    return impfp4::gemv_f4_shape_ok(M, N, K) ? impfp4::gemv_f4_workspace_bytes(M, N, K) : 0;
  return prefill_ws(M, N, K).total;
}

int32_t imp_nvfp4_gemm_plan(int64_t M, int64_t N, int64_t K, const char **kernel) {
  const char *name = nullptr;
  int n = 0;
  if (M >= 1 && N >= 1 && K >= 64 && K % 64 == 0) {
    if (M <= kDecodeMaxM) {
      n = impfp4::gemv_launches(M, N, K, &name);
    } else if (M <= INT32_MAX && N <= INT32_MAX && K <= INT32_MAX) {
      name = "gemm_mxf4_kernel";
      n = 4;  // X amax, X encode, W scale atoms, GEMM
    }
  }
  if (kernel) *kernel = n ? name : nullptr;
  return n;
}

size_t imp_nvfp4_mma_scales_size(int64_t rows, int64_t K) {
  if (rows <= 0 || K <= 0 || K % 64) return 0;
  return impfp4::mma_scale_bytes(rows, K);
}

size_t imp_nvfp4_mma_codes_size(int64_t rows, int64_t K) {
  if (rows <= 0 || K <= 0 || K % 64) return 0;
  return impfp4::mma_code_bytes(rows, K);
}

imp_status imp_nvfp4_prepare_mma(const imp_nvfp4_tensor *t, void *mma_codes, size_t codes_bytes,
                                 void *mma_scales, size_t scales_bytes, void *stream) {
  if (!t || t->rows < 1 || (!mma_codes && !mma_scales)) return IMP_ERR_INVALID_ARG;
  if (t->K <= 0 || t->K % 64) return IMP_ERR_UNSUPPORTED_SHAPE;
  imp_status st = check_tensor(t, t->rows, t->K);
  if (st != IMP_OK) return st;
  if (!aligned16(mma_codes) || !aligned16(mma_scales)) return IMP_ERR_MISALIGNED;
  if (mma_codes && codes_bytes < impfp4::mma_code_bytes(t->rows, t->K))
    return IMP_ERR_WORKSPACE_TOO_SMALL;
  if (mma_scales && scales_bytes < impfp4::mma_scale_bytes(t->rows, t->K))
    return IMP_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (mma_codes)
    e = impfp4::launch_code_relayout(t->codes, t->rows, t->K, static_cast<uint8_t *>(mma_codes), s);
  if (e == cudaSuccess && mma_scales)
    e = impfp4::launch_scale_relayout(t->scales, t->rows, t->K, static_cast<uint8_t *>(mma_scales),
                                      s);
  return from_cuda(e);
}

imp_status imp_nvfp4_quantize_mma(const void *x_bf16, int64_t rows, int64_t K, int64_t ldx,
                                  const imp_nvfp4_tensor *out, int32_t *dev_status,
                                  void *workspace, size_t ws_bytes, void *stream) {
  if (rows < 1 || !x_bf16) return IMP_ERR_INVALID_ARG;
  if (K <= 0 || K % 64) return IMP_ERR_UNSUPPORTED_SHAPE;
  if (ldx < K) return IMP_ERR_INVALID_ARG;
  imp_status st = check_tensor(out, rows, K);
  if (st != IMP_OK) return st;
  if (!aligned16(x_bf16) || ldx % 8) return IMP_ERR_MISALIGNED;
  const size_t need = impfp4::quantize_workspace_bytes(rows, K);
  if (!workspace || ws_bytes < need) return IMP_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned16(workspace)) return IMP_ERR_MISALIGNED;
  return from_cuda(impfp4::launch_quantize_mma(static_cast<const uint16_t *>(x_bf16), rows, K,
                                               ldx, out->codes, out->scales, out->tensor_scale,
                                               dev_status, workspace,
                                               static_cast<cudaStream_t>(stream)));
}

size_t imp_nvfp4_gemm_fp4_workspace_size(int64_t M, int64_t N, int64_t K) {
  if (M < 1 || N < 1 || K <= 0 || K % 64) return 0;
  return impfp4::gemm_mxf4_workspace_bytes(M, N, K);
}

imp_status imp_nvfp4_gemm_fp4(const imp_nvfp4_tensor *xq, const imp_nvfp4_tensor *wq,
                              void *y_bf16, int64_t ldy, int32_t *dev_status, void *workspace,
                              size_t ws_bytes, void *stream) {
  if (!xq || !wq || !y_bf16) return IMP_ERR_INVALID_ARG;
  const int64_t M = xq->rows, N = wq->rows, K = xq->K;
  if (M < 1 || N < 1 || wq->K != K) return IMP_ERR_INVALID_ARG;
  if (K <= 0 || K % 64) return IMP_ERR_UNSUPPORTED_SHAPE;
  if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return IMP_ERR_UNSUPPORTED_SHAPE;
  imp_status st = check_tensor(xq, M, K);
  if (st != IMP_OK) return st;
  st = check_tensor(wq, N, K);
  if (st != IMP_OK) return st;
  if (ldy < N) return IMP_ERR_INVALID_ARG;
  if (!aligned16(y_bf16) || ldy % 8) return IMP_ERR_MISALIGNED;
  if (workspace) {
    if (ws_bytes < impfp4::gemm_mxf4_workspace_bytes(M, N, K)) return IMP_ERR_WORKSPACE_TOO_SMALL;
    if (!aligned16(workspace)) return IMP_ERR_MISALIGNED;
  }
  impfp4::GemmMxf4Plan plan;
  cudaError_t e = impfp4::plan_gemm_mxf4(xq->codes, xq->scales, xq->tensor_scale, wq->codes, true,
                                         wq->scales, wq->tensor_scale, M, N, K,
                                         static_cast<uint16_t *>(y_bf16), ldy, dev_status,
                                         workspace, plan);
  if (e == cudaSuccess) e = impfp4::enqueue_gemm_mxf4(plan, static_cast<cudaStream_t>(stream));
  return from_cuda(e);
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
    if (need && !aligned16(workspace)) return IMP_ERR_MISALIGNED;
    return from_cuda(impfp4::launch_gemv(static_cast<const uint16_t *>(x_bf16), M, K, ldx,
                                         w->codes, w->scales, w->tensor_scale, N,
                                         static_cast<uint16_t *>(y_bf16), ldy, dev_status,
                                         need ? workspace : nullptr, s));
  }
  // Prefill: quantize X (scales straight into the atom layout), lay W's
  // scales out as atoms, then the block-scaled FP4 tensor-core GEMM.  The GEMM
  // is planned first, so a failure returns before anything is enqueued.
  // (A weight in the MMA layout, imp_nvfp4_gemm_mma, skips the W layout.)
  if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return IMP_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(workspace)) return IMP_ERR_MISALIGNED;
  const PrefillWs L = prefill_ws(M, N, K);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  imp_nvfp4_tensor xq = {ws + L.xcodes, ws + L.xsc, reinterpret_cast<float *>(ws + L.sx), M, K};
  imp_nvfp4_tensor wq = {w->codes, ws + L.wsc, w->tensor_scale, N, K};
  impfp4::GemmMxf4Plan plan;
  cudaError_t e = impfp4::plan_gemm_mxf4(xq.codes, xq.scales, xq.tensor_scale, wq.codes, false,
                                         wq.scales, wq.tensor_scale, M, N, K,
                                         static_cast<uint16_t *>(y_bf16), ldy, dev_status,
                                         nullptr, plan);
  if (e != cudaSuccess) return IMP_ERR_CUDA;
  e = impfp4::launch_quantize_mma(static_cast<const uint16_t *>(x_bf16), M, K, ldx, xq.codes,
                                  xq.scales, xq.tensor_scale, dev_status, ws + L.partial, s);
  if (e == cudaSuccess) e = impfp4::launch_scale_relayout(w->scales, N, K, wq.scales, s);
  if (e == cudaSuccess) e = impfp4::enqueue_gemm_mxf4(plan, s);
  return from_cuda(e);
}

imp_status imp_nvfp4_gemm_mma(const void *x_bf16, int64_t M, int64_t K, int64_t ldx,
                              const imp_nvfp4_tensor *w, void *y_bf16, int64_t ldy,
                              int32_t *dev_status, void *workspace, size_t ws_bytes, void *stream) {
  if (M < 0 || !w) return IMP_ERR_INVALID_ARG;
  if (K <= 0 || K % 64) return IMP_ERR_UNSUPPORTED_SHAPE;
  const int64_t N = w->rows;
  if (N < 0 || w->K != K) return IMP_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return IMP_OK;
  imp_status st = check_tensor(w, N, K);
  if (st != IMP_OK) return st;
  if (!x_bf16 || !y_bf16) return IMP_ERR_INVALID_ARG;
  if (ldx < K || ldy < N) return IMP_ERR_INVALID_ARG;
  if (!aligned16(x_bf16) || !aligned16(y_bf16) || ldx % 8 || ldy % 8) return IMP_ERR_MISALIGNED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (M <= kDecodeMaxM) {
    if (!impfp4::gemv_f4_shape_ok(M, N, K)) return IMP_ERR_UNSUPPORTED_SHAPE;
    const size_t need = impfp4::gemv_f4_workspace_bytes(M, N, K);
    if (!workspace || ws_bytes < need) return IMP_ERR_WORKSPACE_TOO_SMALL;
    if (!aligned16(workspace)) return IMP_ERR_MISALIGNED;
    return from_cuda(impfp4::launch_gemv_f4(static_cast<const uint16_t *>(x_bf16), M, K, ldx,
                                            w->codes, w->scales, w->tensor_scale, N,
                                            static_cast<uint16_t *>(y_bf16), ldy, dev_status,
                                            workspace, s, true));
  }
  if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return IMP_ERR_UNSUPPORTED_SHAPE;
  const size_t need = imp_nvfp4_gemm_workspace_size(M, N, K);
  if (!workspace || ws_bytes < need) return IMP_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned16(workspace)) return IMP_ERR_MISALIGNED;
  const PrefillWs L = prefill_ws(M, N, K);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  imp_nvfp4_tensor xq = {ws + L.xcodes, ws + L.xsc, reinterpret_cast<float *>(ws + L.sx), M, K};
  impfp4::GemmMxf4Plan plan;
  cudaError_t e = impfp4::plan_gemm_mxf4(xq.codes, xq.scales, xq.tensor_scale, w->codes, true,
                                         w->scales, w->tensor_scale, M, N, K,
                                         static_cast<uint16_t *>(y_bf16), ldy, dev_status,
                                         nullptr, plan);
  if (e != cudaSuccess) return IMP_ERR_CUDA;
  e = impfp4::launch_quantize_mma(static_cast<const uint16_t *>(x_bf16), M, K, ldx, xq.codes,
                                  xq.scales, xq.tensor_scale, dev_status, ws + L.partial, s);
  if (e == cudaSuccess) e = impfp4::enqueue_gemm_mxf4(plan, s);
  return from_cuda(e);
}

int32_t imp_nvfp4_gemm_mma_swiglu_plan(int64_t M, int64_t N, int64_t K, const char **kernel) {
  const char *k = nullptr;
  const int32_t n = M >= 1 && M <= kDecodeMaxM ? impfp4::gemv_f4_swiglu_launches(M, N, K, &k) : 0;
  if (kernel) *kernel = n ? k : nullptr;
  return n;
}

imp_status imp_nvfp4_gemm_mma_swiglu(const void *gate_bf16, const void *up_bf16, int64_t M,
                                     int64_t K, int64_t ld, const imp_nvfp4_tensor *w,
                                     void *y_bf16, int64_t ldy, int32_t *dev_status,
                                     void *workspace, size_t ws_bytes, void *stream) {
  if (M < 0 || !w) return IMP_ERR_INVALID_ARG;
  if (K <= 0 || K % 64) return IMP_ERR_UNSUPPORTED_SHAPE;
  const int64_t N = w->rows;
  if (N < 0 || w->K != K) return IMP_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return IMP_OK;
  imp_status st = check_tensor(w, N, K);
  if (st != IMP_OK) return st;
  if (!gate_bf16 || !up_bf16 || !y_bf16) return IMP_ERR_INVALID_ARG;
  if (ld < K || ldy < N) return IMP_ERR_INVALID_ARG;
  if (!aligned16(gate_bf16) || !aligned16(up_bf16) || !aligned16(y_bf16) || ld % 8 || ldy % 8)
    return IMP_ERR_MISALIGNED;
  if (M > kDecodeMaxM || !impfp4::gemv_f4_shape_ok(M, N, K)) return IMP_ERR_UNSUPPORTED_SHAPE;
  const size_t need = impfp4::gemv_f4_workspace_bytes(M, N, K);
  if (!workspace || ws_bytes < need) return IMP_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned16(workspace)) return IMP_ERR_MISALIGNED;
  return from_cuda(impfp4::launch_gemv_f4(
      static_cast<const uint16_t *>(gate_bf16), M, K, ld, w->codes, w->scales, w->tensor_scale, N,
      static_cast<uint16_t *>(y_bf16), ldy, dev_status, workspace,
      static_cast<cudaStream_t>(stream), true, static_cast<const uint16_t *>(up_bf16), ld));
}

}  // extern "C"

namespace {

// Kernels one imp_nvfp4_gemm_mma call launches (0: shape rejected).
int32_t mma_plan(int64_t M, int64_t N, int64_t K, const char **kernel) {
  const char *k = nullptr;
  int32_t n = 0;
  if (M >= 1 && N >= 1 && K > 0 && K % 64 == 0) {
    if (M <= kDecodeMaxM) {
      if (impfp4::gemv_f4_shape_ok(M, N, K)) n = impfp4::gemv_f4_launches(M, N, K, &k);
    } else if (M <= INT32_MAX && N <= INT32_MAX && K <= INT32_MAX) {
      n = 3;  // the activation quantizer's two passes and the GEMM
      k = "gemm_mxf4_kernel";
    }
  }
  if (kernel) *kernel = n ? k : nullptr;
  return n;
}

bool grouped_one_pass(int64_t M, int64_t K, const imp_nvfp4_group *g, int32_t n) {
  impfp4::GemvGroup d[IMP_NVFP4_MAX_GROUPS];
  for (int i = 0; i < n; ++i)
    d[i] = {g[i].w.codes, g[i].w.scales, g[i].w.tensor_scale,
            static_cast<uint16_t *>(g[i].y_bf16), g[i].w.rows, g[i].ldy};
  return impfp4::gemv_f4_grouped_ok(M, K, d, n);
}

bool grouped_one_pass_sizes(int64_t M, int64_t K, const int64_t *N, int32_t n) {
  imp_nvfp4_group g[IMP_NVFP4_MAX_GROUPS] = {};
  for (int i = 0; i < n; ++i) g[i].w.rows = N[i];
  return grouped_one_pass(M, K, g, n);
}

}  // namespace

extern "C" {

size_t imp_nvfp4_gemm_grouped_workspace_size(int64_t M, int64_t K, const int64_t *N,
                                             int32_t n_groups) {
  if (!N || n_groups < 1 || n_groups > IMP_NVFP4_MAX_GROUPS || M < 0 || K <= 0) return 0;
  size_t need = 0;
  for (int i = 0; i < n_groups; ++i) {
    if (N[i] < 0) return 0;
    const size_t w = imp_nvfp4_gemm_workspace_size(M, N[i], K);
    need = w > need ? w : need;
  }
  if (grouped_one_pass_sizes(M, K, N, n_groups)) {
    const size_t w = impfp4::gemv_f4_grouped_workspace_bytes(M, K, N, n_groups);
    need = w > need ? w : need;
  }
  return need;
}

int32_t imp_nvfp4_gemm_grouped_plan(int64_t M, int64_t K, const int64_t *N, int32_t n_groups,
                                    const char **kernel) {
  if (kernel) *kernel = nullptr;
  if (!N || n_groups < 1 || n_groups > IMP_NVFP4_MAX_GROUPS) return 0;
  if (grouped_one_pass_sizes(M, K, N, n_groups)) {
    int64_t rows = 0;  // the groups' tiles, scheduled together
    for (int i = 0; i < n_groups; ++i) rows += (N[i] + 127) / 128 * 128;
    const char *k = nullptr;
    const int32_t n = impfp4::gemv_f4_launches(M, rows, K, &k);
    if (kernel) *kernel = k;
    return n;
  }
  int32_t total = 0;
  for (int i = 0; i < n_groups; ++i) {
    const char *k = nullptr;
    const int32_t n = mma_plan(M, N[i], K, &k);
    if (n == 0) return 0;
    total += n;
    if (kernel && !*kernel) *kernel = k;
  }
  return total;
}

imp_status imp_nvfp4_gemm_grouped(const void *x_bf16, int64_t M, int64_t K, int64_t ldx,
                                  const imp_nvfp4_group *groups, int32_t n_groups,
                                  int32_t *dev_status, void *workspace, size_t ws_bytes,
                                  void *stream) {
  if (M < 0 || !groups || n_groups < 1 || n_groups > IMP_NVFP4_MAX_GROUPS) return IMP_ERR_INVALID_ARG;
  if (K <= 0 || K % 64) return IMP_ERR_UNSUPPORTED_SHAPE;
  int64_t N[IMP_NVFP4_MAX_GROUPS];
  for (int i = 0; i < n_groups; ++i) {
    const imp_nvfp4_group &g = groups[i];
    N[i] = g.w.rows;
    if (N[i] < 1 || g.w.K != K) return IMP_ERR_INVALID_ARG;
    imp_status st = check_tensor(&g.w, N[i], K);
    if (st != IMP_OK) return st;
    if (!g.y_bf16 || g.ldy < N[i]) return IMP_ERR_INVALID_ARG;
    if (!aligned16(g.y_bf16) || g.ldy % 8) return IMP_ERR_MISALIGNED;
  }
  if (M == 0) return IMP_OK;
  if (!x_bf16) return IMP_ERR_INVALID_ARG;
  if (ldx < K) return IMP_ERR_INVALID_ARG;
  if (!aligned16(x_bf16) || ldx % 8) return IMP_ERR_MISALIGNED;
  if (imp_nvfp4_gemm_grouped_plan(M, K, N, n_groups, nullptr) == 0) return IMP_ERR_UNSUPPORTED_SHAPE;
  const size_t need = imp_nvfp4_gemm_grouped_workspace_size(M, K, N, n_groups);
  if (!workspace || ws_bytes < need) return IMP_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned16(workspace)) return IMP_ERR_MISALIGNED;
  if (grouped_one_pass(M, K, groups, n_groups)) {
    impfp4::GemvGroup d[IMP_NVFP4_MAX_GROUPS];
    for (int i = 0; i < n_groups; ++i)
      d[i] = {groups[i].w.codes, groups[i].w.scales, groups[i].w.tensor_scale,
              static_cast<uint16_t *>(groups[i].y_bf16), N[i], groups[i].ldy};
    return from_cuda(impfp4::launch_gemv_f4_grouped(static_cast<const uint16_t *>(x_bf16), M, K,
                                                    ldx, d, n_groups, dev_status, workspace,
                                                    static_cast<cudaStream_t>(stream)));
  }
  // one call per weight, in order, sharing the workspace
  for (int i = 0; i < n_groups; ++i) {
    const imp_status st = imp_nvfp4_gemm_mma(x_bf16, M, K, ldx, &groups[i].w, groups[i].y_bf16,
                                             groups[i].ldy, dev_status, workspace, ws_bytes, stream);
    if (st != IMP_OK) return st;
  }
  return IMP_OK;
}

}  // extern "C"

// ---- decode chain ------------------------------------------------------------------

namespace {
struct ChainResolved {
  impfp4::GemvGroup g[IMP_NVFP4_MAX_CHAIN][IMP_NVFP4_MAX_GROUPS];
  int64_t N[IMP_NVFP4_MAX_CHAIN][IMP_NVFP4_MAX_GROUPS];
  impfp4::ChainLink l[IMP_NVFP4_MAX_CHAIN];
};

// Bytes spanned by M rows of `cols` bf16 elements at stride ld.
uintptr_t span_bytes(int64_t M, int64_t ld, int64_t cols) {
  return (uintptr_t)(((M - 1) * ld + cols) * 2);
}
bool overlap(const void *a, uintptr_t na, const void *b, uintptr_t nb) {
  const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
  return pa < pb + nb && pb < pa + na;
}

// The links with each X resolved (the NULL form reads the previous link's
// first output).  sizes_only: look at K and the weights' rows alone.
imp_status resolve_chain(int64_t M, const imp_nvfp4_chain_link *links, int32_t n, bool sizes_only,
                         ChainResolved &r) {
  if (M < 0 || !links || n < 1 || n > IMP_NVFP4_MAX_CHAIN) return IMP_ERR_INVALID_ARG;
  for (int c = 0; c < n; ++c) {
    const imp_nvfp4_chain_link &L = links[c];
    if (!L.groups || L.n_groups < 1 || L.n_groups > IMP_NVFP4_MAX_GROUPS) return IMP_ERR_INVALID_ARG;
    const int64_t K = L.groups[0].w.K;
    if (K <= 0 || K % 64) return IMP_ERR_UNSUPPORTED_SHAPE;
    for (int i = 0; i < L.n_groups; ++i) {
      const imp_nvfp4_group &g = L.groups[i];
      const int64_t N = g.w.rows;
      if (N < 1 || g.w.K != K) return IMP_ERR_INVALID_ARG;
      if (!sizes_only) {
        const imp_status st = check_tensor(&g.w, N, K);
        if (st != IMP_OK) return st;
        if (!g.y_bf16 || g.ldy < N) return IMP_ERR_INVALID_ARG;
        if (!aligned16(g.y_bf16) || g.ldy % 8) return IMP_ERR_MISALIGNED;
      }
      r.N[c][i] = N;
      r.g[c][i] = {g.w.codes, g.w.scales, g.w.tensor_scale, static_cast<uint16_t *>(g.y_bf16), N,
                   g.ldy};
    }
    const uint16_t *x = static_cast<const uint16_t *>(L.x_bf16);
    int64_t ldx = L.ldx;
    const uint16_t *x2 = nullptr;
    int64_t ldx2 = 0;
    const bool dep = x == nullptr;
    if (L.x_swiglu && !dep) return IMP_ERR_INVALID_ARG;
    if (dep) {
      if (c == 0 || K != links[c - 1].groups[0].w.rows) return IMP_ERR_INVALID_ARG;
      x = static_cast<const uint16_t *>(links[c - 1].groups[0].y_bf16);
      ldx = links[c - 1].groups[0].ldy;
      if (L.x_swiglu) {  // X = silu(previous groups[0] output) * previous groups[1] output
        if (links[c - 1].n_groups < 2 || links[c - 1].groups[1].w.rows != K)
          return IMP_ERR_INVALID_ARG;
        x2 = static_cast<const uint16_t *>(links[c - 1].groups[1].y_bf16);
        ldx2 = links[c - 1].groups[1].ldy;
      }
    } else if (!sizes_only && M > 0) {
      if (ldx < K) return IMP_ERR_INVALID_ARG;
      if (!aligned16(x) || ldx % 8) return IMP_ERR_MISALIGNED;
    }
    r.l[c] = impfp4::ChainLink{r.g[c], L.n_groups, x, ldx, K, dep, x2, ldx2};
  }
  if (sizes_only || M == 0) return IMP_OK;
  // links run concurrently on different SMs: no output may overlap another
  // link's output or any explicit X
  for (int c = 0; c < n; ++c)
    for (int i = 0; i < links[c].n_groups; ++i) {
      const imp_nvfp4_group &g = links[c].groups[i];
      const uintptr_t ny = span_bytes(M, g.ldy, g.w.rows);
      for (int d = 0; d < n; ++d) {
        if (links[d].x_bf16 &&
            overlap(g.y_bf16, ny, links[d].x_bf16, span_bytes(M, links[d].ldx, r.l[d].K)))
          return IMP_ERR_INVALID_ARG;
        if (d == c) continue;
        for (int j = 0; j < links[d].n_groups; ++j) {
          const imp_nvfp4_group &h = links[d].groups[j];
          if (overlap(g.y_bf16, ny, h.y_bf16, span_bytes(M, h.ldy, h.w.rows)))
            return IMP_ERR_INVALID_ARG;
        }
      }
    }
  return IMP_OK;
}
}  // namespace

extern "C" {

size_t imp_nvfp4_gemm_chain_workspace_size(int64_t M, const imp_nvfp4_chain_link *links,
                                           int32_t n_links) {
  ChainResolved r;
  if (resolve_chain(M, links, n_links, true, r) != IMP_OK) return 0;
  size_t need = 0;
  for (int c = 0; c < n_links; ++c) {
    const size_t w = imp_nvfp4_gemm_grouped_workspace_size(M, r.l[c].K, r.N[c], links[c].n_groups);
    need = w > need ? w : need;
  }
  if (M >= 1 && impfp4::gemv_f4_chain_ok(M, r.l, n_links)) {
    const size_t w = impfp4::gemv_f4_chain_workspace_bytes(M, r.l, n_links);
    need = w > need ? w : need;
  }
  return need;
}

int32_t imp_nvfp4_gemm_chain_plan(int64_t M, const imp_nvfp4_chain_link *links, int32_t n_links) {
  ChainResolved r;
  if (resolve_chain(M, links, n_links, true, r) != IMP_OK) return 0;
  return M >= 1 && impfp4::gemv_f4_chain_ok(M, r.l, n_links) ? 1 : 0;
}

imp_status imp_nvfp4_gemm_chain(int64_t M, const imp_nvfp4_chain_link *links, int32_t n_links,
                                int32_t *dev_status, void *workspace, size_t ws_bytes,
                                void *stream) {
  ChainResolved r;
  const imp_status st = resolve_chain(M, links, n_links, false, r);
  if (st != IMP_OK) return st;
  if (M == 0) return IMP_OK;
  const size_t need = imp_nvfp4_gemm_chain_workspace_size(M, links, n_links);
  if (!workspace || ws_bytes < need) return IMP_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned16(workspace)) return IMP_ERR_MISALIGNED;
  if (impfp4::gemv_f4_chain_ok(M, r.l, n_links))
    return from_cuda(impfp4::launch_gemv_f4_chain(M, r.l, n_links, dev_status, workspace,
                                                  static_cast<cudaStream_t>(stream)));
  // one grouped call per link, in order (every link checked before any
  // runs); a link on silu(g) * u runs its groups one by one
  for (int c = 0; c < n_links; ++c) {
    if (r.l[c].x2) {
      if (r.l[c].ldx2 != r.l[c].ldx) return IMP_ERR_UNSUPPORTED_SHAPE;
      for (int i = 0; i < links[c].n_groups; ++i)
        if (imp_nvfp4_gemm_mma_swiglu_plan(M, r.N[c][i], r.l[c].K, nullptr) == 0)
          return IMP_ERR_UNSUPPORTED_SHAPE;
    } else if (imp_nvfp4_gemm_grouped_plan(M, r.l[c].K, r.N[c], links[c].n_groups, nullptr) == 0) {
      return IMP_ERR_UNSUPPORTED_SHAPE;
    }
  }
  for (int c = 0; c < n_links; ++c) {
    imp_status s = IMP_OK;
    if (r.l[c].x2) {
      for (int i = 0; i < links[c].n_groups && s == IMP_OK; ++i)
        s = imp_nvfp4_gemm_mma_swiglu(r.l[c].x, r.l[c].x2, M, r.l[c].K, r.l[c].ldx,
                                      &links[c].groups[i].w, links[c].groups[i].y_bf16,
                                      links[c].groups[i].ldy, dev_status, workspace, ws_bytes,
                                      stream);
    } else {
      s = imp_nvfp4_gemm_grouped(r.l[c].x, M, r.l[c].K, r.l[c].ldx, links[c].groups,
                                 links[c].n_groups, dev_status, workspace, ws_bytes, stream);
    }
    if (s != IMP_OK) return s;
  }
  return IMP_OK;
}

// ---- MXFP4 and FP8 weights ----------------------------------------------------

imp_status imp_mxfp4_quantize(const void *x_bf16, int64_t rows, int64_t K, int64_t ldx,
                              const imp_mxfp4_tensor *out, int32_t *dev_status, void *stream) {
  if (rows < 1 || K <= 0 || !out || !x_bf16) return IMP_ERR_INVALID_ARG;
  if (K % 32) return IMP_ERR_UNSUPPORTED_SHAPE;
  if (ldx < K || out->rows != rows || out->K != K || !out->codes || !out->scales)
    return IMP_ERR_INVALID_ARG;
  if (!aligned16(x_bf16) || ldx % 8 || !aligned16(out->codes)) return IMP_ERR_MISALIGNED;
  return from_cuda(impfp4::launch_mx_quantize(static_cast<const uint16_t *>(x_bf16), rows, K, ldx,
                                              out->codes, out->scales, dev_status,
                                              static_cast<cudaStream_t>(stream)));
}

size_t imp_mxfp4_to_nvfp4_workspace_size(void) { return 16; }

imp_status imp_mxfp4_to_nvfp4(const imp_mxfp4_tensor *in, const imp_nvfp4_tensor *out,
                              int32_t *dev_status, void *workspace, size_t ws_bytes,
                              void *stream) {
  if (!in || !out || !in->codes || !in->scales) return IMP_ERR_INVALID_ARG;
  if (in->rows < 1 || in->K <= 0) return IMP_ERR_INVALID_ARG;
  if (in->K % 64) return IMP_ERR_UNSUPPORTED_SHAPE;
  imp_status st = check_tensor(out, in->rows, in->K);
  if (st != IMP_OK) return st;
  if (!aligned16(in->codes)) return IMP_ERR_MISALIGNED;
  if (!workspace || ws_bytes < imp_mxfp4_to_nvfp4_workspace_size()) return IMP_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned4(workspace)) return IMP_ERR_MISALIGNED;
  return from_cuda(impfp4::launch_mx_to_nvfp4(in->codes, in->scales, in->rows, in->K, out->codes,
                                              out->scales, out->tensor_scale, dev_status,
                                              workspace, static_cast<cudaStream_t>(stream)));
}

size_t imp_fp8_quantize_workspace_size(int64_t rows, int64_t K) {
  if (rows <= 0 || K <= 0) return 0;
  return impfp4::quantize_workspace_bytes(rows, K);
}

imp_status imp_fp8_quantize(const void *x_bf16, int64_t rows, int64_t K, int64_t ldx,
                            const imp_fp8_tensor *out, int32_t *dev_status, void *workspace,
                            size_t ws_bytes, void *stream) {
  if (rows < 1 || K <= 0 || !out || !x_bf16) return IMP_ERR_INVALID_ARG;
  if (K % 16) return IMP_ERR_UNSUPPORTED_SHAPE;
  if (ldx < K || out->rows != rows || out->K != K || !out->codes || !out->tensor_scale)
    return IMP_ERR_INVALID_ARG;
  if (!aligned16(x_bf16) || ldx % 8 || !aligned16(out->codes) || !aligned4(out->tensor_scale))
    return IMP_ERR_MISALIGNED;
  if (!workspace || ws_bytes < impfp4::quantize_workspace_bytes(rows, K))
    return IMP_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned16(workspace)) return IMP_ERR_MISALIGNED;
  return from_cuda(impfp4::launch_fp8_quantize(static_cast<const uint16_t *>(x_bf16), rows, K, ldx,
                                               out->codes, out->tensor_scale, dev_status,
                                               workspace, static_cast<cudaStream_t>(stream)));
}

size_t imp_fp8_gemm_workspace_size(int64_t M, int64_t N, int64_t K) {
  if (M < 1 || M > kDecodeMaxM || !impfp4::gemv_fp8_shape_ok(M, N, K)) return 0;
  return impfp4::gemv_fp8_workspace_bytes(N, K);
}

int32_t imp_fp8_gemm_plan(int64_t M, int64_t N, int64_t K, const char **kernel) {
  const bool ok = M >= 1 && M <= kDecodeMaxM && impfp4::gemv_fp8_shape_ok(M, N, K);
  if (kernel) *kernel = ok ? "gemv_f4r_kernel" : nullptr;
  return ok ? impfp4::gemv_fp8_launches(M) : 0;
}

imp_status imp_fp8_gemm(const void *x_bf16, int64_t M, int64_t K, int64_t ldx,
                        const imp_fp8_tensor *w, void *y_bf16, int64_t ldy, int32_t *dev_status,
                        void *workspace, size_t ws_bytes, void *stream) {
  if (M < 0 || !w) return IMP_ERR_INVALID_ARG;
  const int64_t N = w->rows;
  if (N < 0 || w->K != K || K <= 0) return IMP_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return IMP_OK;
  if (!w->codes || !w->tensor_scale || !x_bf16 || !y_bf16) return IMP_ERR_INVALID_ARG;
  if (ldx < K || ldy < N) return IMP_ERR_INVALID_ARG;
  if (M > kDecodeMaxM || !impfp4::gemv_fp8_shape_ok(M, N, K)) return IMP_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(x_bf16) || !aligned16(y_bf16) || !aligned16(w->codes) ||
      !aligned4(w->tensor_scale) || ldx % 8 || ldy % 8)
    return IMP_ERR_MISALIGNED;
  const size_t need = impfp4::gemv_fp8_workspace_bytes(N, K);
  if (!workspace || ws_bytes < need) return IMP_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned16(workspace)) return IMP_ERR_MISALIGNED;
  return from_cuda(impfp4::launch_gemv_fp8(static_cast<const uint16_t *>(x_bf16), M, K, ldx,
                                           w->codes, w->tensor_scale, N,
                                           static_cast<uint16_t *>(y_bf16), ldy, dev_status,
                                           workspace, static_cast<cudaStream_t>(stream)));
}

// ---- fused prefill MLP pieces ---------------------------------------------------

size_t imp_nvfp4_gemm_swiglu_workspace_size(int64_t M, int64_t N, int64_t K) {
  if (M <= kDecodeMaxM || N < 1 || K <= 0 || K % 64) return 0;
  return prefill_ws(M, N, K).total;
}

imp_status imp_nvfp4_gemm_swiglu(const void *x_bf16, int64_t M, int64_t K, int64_t ldx,
                                 const imp_nvfp4_tensor *w_gate, const imp_nvfp4_tensor *w_up,
                                 void *h_bf16, int64_t ldh, uint32_t *h_amax,
                                 int32_t *dev_status, void *workspace, size_t ws_bytes,
                                 void *stream) {
  if (M < 0 || !w_gate || !w_up) return IMP_ERR_INVALID_ARG;
  if (K <= 0 || K % 64) return IMP_ERR_UNSUPPORTED_SHAPE;
  const int64_t N = w_gate->rows;
  if (N < 1 || w_up->rows != N || w_gate->K != K || w_up->K != K) return IMP_ERR_INVALID_ARG;
  imp_status st = check_tensor(w_gate, N, K);
  if (st == IMP_OK) st = check_tensor(w_up, N, K);
  if (st != IMP_OK) return st;
  if (M == 0) return IMP_OK;
  if (!x_bf16 || !h_bf16 || !h_amax || ldx < K || ldh < N) return IMP_ERR_INVALID_ARG;
  if (M <= kDecodeMaxM || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX)
    return IMP_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(x_bf16) || !aligned16(h_bf16) || !aligned4(h_amax) || ldx % 8 || ldh % 8)
    return IMP_ERR_MISALIGNED;
  const size_t need = imp_nvfp4_gemm_swiglu_workspace_size(M, N, K);
  if (!workspace || ws_bytes < need) return IMP_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned16(workspace)) return IMP_ERR_MISALIGNED;
  const PrefillWs L = prefill_ws(M, N, K);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  imp_nvfp4_tensor xq = {ws + L.xcodes, ws + L.xsc, reinterpret_cast<float *>(ws + L.sx), M, K};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  impfp4::GemmMxf4Plan plan;
  cudaError_t e = impfp4::plan_gemm_mxf4_swiglu(
      xq.codes, xq.scales, xq.tensor_scale, w_gate->codes, w_gate->scales, w_gate->tensor_scale,
      w_up->codes, w_up->scales, w_up->tensor_scale, M, N, K, static_cast<uint16_t *>(h_bf16), ldh,
      h_amax, dev_status, plan);
  if (e != cudaSuccess) return IMP_ERR_CUDA;
  e = cudaMemsetAsync(h_amax, 0, sizeof(uint32_t), s);
  if (e == cudaSuccess)
    e = impfp4::launch_quantize_mma(static_cast<const uint16_t *>(x_bf16), M, K, ldx, xq.codes,
                                    xq.scales, xq.tensor_scale, dev_status, ws + L.partial, s);
  if (e == cudaSuccess) e = impfp4::enqueue_gemm_mxf4(plan, s);
  return from_cuda(e);
}

imp_status imp_nvfp4_quantize_mma_amax(const void *x_bf16, int64_t rows, int64_t K, int64_t ldx,
                                       const uint32_t *amax, const imp_nvfp4_tensor *out,
                                       int32_t *dev_status, void *stream) {
  (void)dev_status;
  if (rows < 1 || K <= 0 || !x_bf16 || !amax) return IMP_ERR_INVALID_ARG;
  if (K % 64) return IMP_ERR_UNSUPPORTED_SHAPE;
  if (ldx < K) return IMP_ERR_INVALID_ARG;
  if (!out || out->rows != rows || out->K != K || !out->codes || !out->scales ||
      !out->tensor_scale)
    return IMP_ERR_INVALID_ARG;
  if (!aligned16(x_bf16) || ldx % 8 || !aligned16(out->codes) || !aligned4(amax) ||
      !aligned4(out->tensor_scale))
    return IMP_ERR_MISALIGNED;
  return from_cuda(impfp4::launch_encode_with_amax(static_cast<const uint16_t *>(x_bf16), rows, K,
                                                   ldx, amax, out->codes, out->scales,
                                                   out->tensor_scale, true,
                                                   static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
