// Decode-path NVFP4 GEMV / skinny GEMM: Y[M][N] = X[M][K] * W^T for M <= 16.
//
// This file holds the dispatch between the decode kernels (launch_gemv,
// choose_path: the FP4 tensor-core kernel of gemv_f4.cu, the f16
// tensor-core kernel of gemv_tc.cu) and the CUDA-core kernel below, which
// takes the shapes neither tensor-core kernel accepts (K beyond the f16
// kernel's register-resident X, up to 61440, when the FP4 kernel's shape
// rules are not met).
//
// Decode is bandwidth-bound: every weight byte is read once per step and the
// arithmetic is trivial next to it (imp README, "How it works"; "1. The big
// picture", section "The most important number in this book").  The
// CUDA-core kernel is therefore built around streaming W at HBM speed:
//
//  * Persistent grid, one CTA per SM; CTA c owns the contiguous row range
//    [N*c/G, N*(c+1)/G) of W, so the load is balanced to within one row.
//  * A producer warp streams whole rows of W (codes, and scales when K is a
//    multiple of 256) into a ring of shared-memory stages with 1-D bulk
//    copies (cp.async.bulk, completion counted on an mbarrier).  Rows of the
//    [N][K/2] code array are contiguous, so a stage of RS rows is one copy.
//  * Consumer threads own fixed 32-element chunks of K (chunk c = t + j*P for
//    the P threads sharing a row) and keep the matching slice of X in
//    registers as f16 -- the same registers serve every row the CTA streams.
//    X is rescaled per chunk by a power of two so the f16 copy is exact for
//    any bf16 magnitude (the factor is undone in fp32 at the end of the row).
//  * Decode: cvt.rn.f16x2.e2m1x2 turns each byte into two f16 values; each
//    product with X is accumulated in fp32 by fma.rn.f32.f16 (the product of
//    two f16 values is exact in fp32).  A block's sum is scaled by its E4M3
//    scale (cvt.rn.f16x2.e4m3x2) in fp32.
//  * Row sums: warp shuffle reduction, then a fixed-order sum of the per-warp
//    partials in shared memory, times the tensor scale, rounded to bf16.
//    The order never depends on timing, so results are bitwise reproducible.
#include "gemv.cuh"

namespace impfp4 {

namespace {

constexpr int kProducerThreads = 32;
constexpr int kMaxStages = 8;
constexpr size_t kSmemBudget = 200 * 1024;
// mbarriers (full[8], empty[8]), the abort flag, padding to 16 bytes.
constexpr size_t kHeadBytes = 2 * kMaxStages * sizeof(uint64_t) + 16;

// Largest block (threads) an instantiation is compiled for: the X registers
// grow with CPT * MT, so fewer threads fit the 64K-register file.
__host__ __device__ constexpr int max_threads_for(int cpt, int mt) {
  return cpt * mt <= 1 ? 1024 : cpt * mt <= 2 ? 768 : cpt * mt <= 4 ? 512 : 384;
}

struct GemvArgs {
  const uint16_t *x;
  int64_t ldx;
  int M;  // rows of X handled by this launch (<= MT)
  const uint8_t *codes;
  const uint8_t *scales;
  const float *tensor_scale;
  uint16_t *y;
  int64_t ldy;
  int64_t N, K;
  int32_t *status;
  int rows_per_stage;  // RS
  int nstages;         // NS
  int threads_per_row; // P, multiple of 32
  int row_groups;      // RG
  int scales_bulk;     // 1: scales staged by bulk copy; 0: read from global
  uint32_t stage_bytes, codes_stage_bytes;
};

__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Two fp32 accumulations acc += a.lo*b.lo, acc2 += a.hi*b.hi of f16x2 words.
__device__ __forceinline__ void fma2_f16_f32(uint32_t a, uint32_t b, float &acc0, float &acc1) {
  asm("{\n.reg .b16 a0, a1, b0, b1;\nmov.b32 {a0, a1}, %2;\nmov.b32 {b0, b1}, %3;\n"
      "fma.rn.f32.f16 %0, a0, b0, %0;\nfma.rn.f32.f16 %1, a1, b1, %1;\n}"
      : "+f"(acc0), "+f"(acc1)
      : "r"(a), "r"(b));
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&h);
}

template <int CPT, int MT>
__global__ void __launch_bounds__(max_threads_for(CPT, MT), 1) gemv_kernel(const GemvArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int NS = a.nstages, RS = a.rows_per_stage, P = a.threads_per_row, RG = a.row_groups;
  const int NWK = P / 32;  // warps sharing a row
  const int n_consumer_warps = (P * RG) / 32;
  const int64_t KH = a.K / 2, KB = a.K / 16, C = a.K / 32;

  uint64_t *full = reinterpret_cast<uint64_t *>(smem);
  uint64_t *empty = full + kMaxStages;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + kMaxStages);
  float *red = reinterpret_cast<float *>(smem + 2 * kMaxStages * sizeof(uint64_t) + 16);  // [NS][RS][MT][NWK]
  const size_t red_bytes = (size_t)NS * RS * MT * NWK * sizeof(float);
  uint8_t *stages = smem + kHeadBytes + ((red_bytes + 127) / 128) * 128;

  const int64_t G = gridDim.x;
  const int64_t row_begin = a.N * (int64_t)blockIdx.x / G;
  const int64_t row_end = a.N * ((int64_t)blockIdx.x + 1) / G;
  const int64_t n_rows = row_end - row_begin;
  const int64_t n_st = ceil_div(n_rows, RS);

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], n_consumer_warps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (threadIdx.x < kProducerThreads) {
    // ---------------- producer: one thread streams stages ----------------
    if (threadIdx.x != 0) return;
    int64_t issued = 0;
    bool ok = true;
    for (int64_t i = 0; i < n_st; ++i) {
      const int s = (int)(i % NS);
      if (i >= NS && !mbar_wait_bounded(&empty[s], (uint32_t)(((i / NS) - 1) & 1), a.status)) {
        ok = false;
        break;
      }
      const int64_t r0 = row_begin + i * RS;
      const int64_t rows_i = min((int64_t)RS, row_end - r0);
      const uint32_t cbytes = (uint32_t)(rows_i * KH);
      const uint32_t sbytes = a.scales_bulk ? (uint32_t)(rows_i * KB) : 0u;
      uint8_t *st = stages + (size_t)s * a.stage_bytes;
      mbar_arrive_expect_tx(&full[s], cbytes + sbytes);
      bulk_g2s(st, a.codes + r0 * KH, cbytes, &full[s]);
      if (sbytes) bulk_g2s(st + a.codes_stage_bytes, a.scales + r0 * KB, sbytes, &full[s]);
      ++issued;
    }
    if (!ok) {
      // Drain: every issued copy must land before this CTA's shared memory
      // is released.  Stage s's last issued copy completes phase (i / NS).
      for (int64_t i = (issued > NS ? issued - NS : 0); i < issued; ++i)
        mbar_wait_bounded(&full[i % NS], (uint32_t)((i / NS) & 1), a.status);
    }
    return;
  }

  // ---------------- consumers ----------------
  const int ct = threadIdx.x - kProducerThreads;
  const int rg = ct / P;
  const int t = ct - rg * P;
  const int lane = threadIdx.x & 31;
  const int wk = t / 32;  // warp index within the row group

  // Load this thread's X chunks into registers as f16, rescaled by 2^sh per
  // (row of X, chunk) so the largest magnitude of the chunk lies in
  // [2^14, 2^15): exact for every bf16 value within 31 binades of the max.
  uint32_t xh[MT][CPT][16];
  float xinv[MT][CPT];
#pragma unroll
  for (int m = 0; m < MT; ++m) {
#pragma unroll
    for (int j = 0; j < CPT; ++j) {
      const int64_t c = t + (int64_t)j * P;
      xinv[m][j] = 0.0f;
#pragma unroll
      for (int i = 0; i < 16; ++i) xh[m][j][i] = 0u;
      if (c < C && m < a.M) {
        const uint4 *src = reinterpret_cast<const uint4 *>(a.x + (int64_t)m * a.ldx + c * 32);
        uint32_t w[16];
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const uint4 q = __ldg(src + v);
          w[4 * v] = q.x; w[4 * v + 1] = q.y; w[4 * v + 2] = q.z; w[4 * v + 3] = q.w;
        }
        uint32_t mx = 0;
#pragma unroll
        for (int i = 0; i < 16; ++i) mx = __vmaxu2(mx, w[i] & 0x7FFF7FFFu);
        const float amax = bf16_bits_to_f32(max(mx & 0xFFFFu, mx >> 16));
        int sh = 0;
        if (amax > 0.0f) {
          int e;
          frexpf(amax, &e);  // amax in [2^(e-1), 2^e)
          sh = 15 - e;       // amax * 2^sh in [2^14, 2^15)
        }
        xinv[m][j] = ldexpf(1.0f, -sh);
#pragma unroll
        for (int i = 0; i < 16; ++i)
          xh[m][j][i] = pack_f16x2(ldexpf(bf16_bits_to_f32(w[i] & 0xFFFFu), sh),
                                   ldexpf(bf16_bits_to_f32(w[i] >> 16), sh));
      }
    }
  }
  const float ts = *a.tensor_scale;

  for (int64_t i = 0; i < n_st; ++i) {
    const int s = (int)(i % NS);
    // A warp whose wait gives up still meets the others at the named barrier
    // below, so no consumer can be left waiting there; all leave together.
    // warp-uniform: the shuffles below need all 32 lanes
    const bool ready =
        __all_sync(0xFFFFFFFFu, mbar_wait_bounded(&full[s], (uint32_t)((i / NS) & 1), a.status));
    if (!ready) *abort_flag = 1;
    const int64_t r0 = row_begin + i * RS;
    const int rows_i = (int)min((int64_t)RS, row_end - r0);
    const uint8_t *st_codes = stages + (size_t)s * a.stage_bytes;
    const uint8_t *st_scales = st_codes + a.codes_stage_bytes;
    float *red_s = red + (size_t)s * RS * MT * NWK;

    for (int r = ready ? rg : rows_i; r < rows_i; r += RG) {
      float acc[MT][CPT];
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int j = 0; j < CPT; ++j) acc[m][j] = 0.0f;
#pragma unroll
      for (int j = 0; j < CPT; ++j) {
        const int64_t c = t + (int64_t)j * P;
        if (c < C) {
          const uint4 cw = *reinterpret_cast<const uint4 *>(st_codes + r * KH + c * 16);
          uint32_t sc2;
          if (a.scales_bulk)
            sc2 = *reinterpret_cast<const uint16_t *>(st_scales + r * KB + c * 2);
          else
            sc2 = __ldg(reinterpret_cast<const uint16_t *>(a.scales + (r0 + r) * KB + c * 2));
          const uint32_t dsc = e4m3x2_to_f16x2(sc2);
          const float d0 = f16lo_to_f32(dsc), d1 = f16hi_to_f32(dsc);
          uint32_t h[16];
          e2m1x8_to_f16x2x4(cw.x, *reinterpret_cast<uint32_t(*)[4]>(&h[0]));
          e2m1x8_to_f16x2x4(cw.y, *reinterpret_cast<uint32_t(*)[4]>(&h[4]));
          e2m1x8_to_f16x2x4(cw.z, *reinterpret_cast<uint32_t(*)[4]>(&h[8]));
          e2m1x8_to_f16x2x4(cw.w, *reinterpret_cast<uint32_t(*)[4]>(&h[12]));
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            float b0e = 0.f, b0o = 0.f, b1e = 0.f, b1o = 0.f;
#pragma unroll
            for (int q = 0; q < 8; ++q) fma2_f16_f32(h[q], xh[m][j][q], b0e, b0o);
#pragma unroll
            for (int q = 8; q < 16; ++q) fma2_f16_f32(h[q], xh[m][j][q], b1e, b1o);
            acc[m][j] = fmaf(b0e + b0o, d0, acc[m][j]);
            acc[m][j] = fmaf(b1e + b1o, d1, acc[m][j]);
          }
        }
      }
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        float v = 0.0f;
#pragma unroll
        for (int j = 0; j < CPT; ++j) v = fmaf(acc[m][j], xinv[m][j], v);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
        if (lane == 0) red_s[((size_t)r * MT + m) * NWK + wk] = v;
      }
    }
    named_barrier_sync(1, n_consumer_warps * 32);
    if (*abort_flag) return;
    for (int o = ct; o < rows_i * MT; o += n_consumer_warps * 32) {
      const int r = o / MT, m = o - r * MT;
      if (m < a.M) {
        float v = 0.0f;
        for (int w = 0; w < NWK; ++w) v += red_s[((size_t)r * MT + m) * NWK + w];
        v *= ts;
        a.y[(int64_t)m * a.ldy + r0 + r] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
}

struct Plan {
  int MT, CPT, P, RG, RS, NS, threads;
  int scales_bulk;
  uint32_t stage_bytes, codes_stage_bytes;
  size_t smem;
};

// Choose the launch shape for one pass of MT rows of X.
bool make_plan(int MT, int64_t N, int64_t K, Plan &p) {
  const int64_t C = K / 32;
  p.MT = MT;
  const int max_cpt = 8 / MT < 4 ? 8 / MT : 4;
  int best_cpt = -1;
  int64_t best_P = 0;
  double best_waste = 1e9;
  for (int cpt = 1; cpt <= max_cpt; ++cpt) {
    int64_t P = ceil_div(ceil_div(C, cpt), 32) * 32;
    if (P + kProducerThreads > max_threads_for(cpt, MT)) continue;
    const double waste = (double)(P * cpt - C) / (double)(P * cpt);
    // prefer fewer registers (smaller cpt) unless it wastes lanes
    if (waste + 0.02 * cpt < best_waste) {
      best_waste = waste + 0.02 * cpt;
      best_cpt = cpt;
      best_P = P;
    }
  }
  if (best_cpt < 0) return false;
  p.CPT = best_cpt;
  p.P = (int)best_P;
  const int warps_per_row = p.P / 32;
  int RG = 16 / warps_per_row;
  if (RG < 1) RG = 1;
  while (RG > 1 && RG * p.P + kProducerThreads > max_threads_for(p.CPT, MT)) --RG;
  p.RG = RG;
  p.threads = kProducerThreads + p.RG * p.P;
  p.scales_bulk = (K % 256 == 0) ? 1 : 0;
  const int64_t row_bytes = K / 2 + (p.scales_bulk ? K / 16 : 0);
  int64_t RS = (24 * 1024) / row_bytes;
  if (RS < p.RG) RS = p.RG;
  if (RS < 1) RS = 1;
  if (RS > 64) RS = 64;
  const int64_t rows_per_cta = ceil_div(N, num_sms());
  if (RS > rows_per_cta) RS = rows_per_cta < 1 ? 1 : rows_per_cta;
  p.RS = (int)RS;
  p.codes_stage_bytes = (uint32_t)(ceil_div(RS * (K / 2), 128) * 128);
  const uint32_t scale_bytes = p.scales_bulk ? (uint32_t)(ceil_div(RS * (K / 16), 128) * 128) : 0u;
  p.stage_bytes = p.codes_stage_bytes + scale_bytes;
  const size_t head = kHeadBytes;
  int NS = kMaxStages;
  while (NS > 2) {
    const size_t red = (size_t)NS * p.RS * MT * (p.P / 32) * sizeof(float);
    if (head + ceil_div(red, 128) * 128 + (size_t)NS * p.stage_bytes <= kSmemBudget) break;
    --NS;
  }
  p.NS = NS;
  const size_t red = (size_t)NS * p.RS * MT * (p.P / 32) * sizeof(float);
  p.smem = head + ceil_div(red, 128) * 128 + (size_t)NS * p.stage_bytes;
  return p.smem <= kSmemBudget + 16 * 1024;
}

template <int CPT, int MT>
cudaError_t launch_one(const GemvArgs &a, const Plan &p, int grid, cudaStream_t stream) {
  auto kern = gemv_kernel<CPT, MT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, p.threads, p.smem, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t dispatch(const GemvArgs &a, const Plan &p, int grid, cudaStream_t stream) {
#define IMPFP4_CASE(cpt, mt) \
  if (p.CPT == cpt && p.MT == mt) return launch_one<cpt, mt>(a, p, grid, stream);
  IMPFP4_CASE(1, 1) IMPFP4_CASE(2, 1) IMPFP4_CASE(3, 1) IMPFP4_CASE(4, 1)
  IMPFP4_CASE(1, 2) IMPFP4_CASE(2, 2) IMPFP4_CASE(3, 2) IMPFP4_CASE(4, 2)
  IMPFP4_CASE(1, 4) IMPFP4_CASE(2, 4)
  IMPFP4_CASE(1, 8)
#undef IMPFP4_CASE
  return cudaErrorInvalidConfiguration;
}

// Rows of X per pass: the largest tile in {8, 4, 2, 1} that has a launch
// plan for this K, not above the rows left (rounded up to a power of two).
int pass_tile(int64_t M_left, int64_t N, int64_t K, Plan &p) {
  int want = M_left >= 5 ? 8 : M_left >= 3 ? 4 : (int)M_left;
  for (int mt = want; mt >= 1; mt /= 2)
    if (make_plan(mt, N, K, p)) return mt;
  return 0;
}

}  // namespace

namespace {

// CUDA-core passes needed for M rows of X (0: no plan fits).
int cuda_core_passes(int64_t M, int64_t N, int64_t K) {
  int passes = 0;
  for (int64_t m0 = 0; m0 < M; ++passes) {
    Plan p;
    const int MT = pass_tile(M - m0, N, K, p);
    if (MT == 0) return 0;
    m0 += MT;
  }
  return passes;
}

enum class DecodePath { kNone, kFp4, kF16, kCudaCore };

// Measured on GB300 (back-to-back calls, weights from HBM): wherever the
// FP4 path takes the shape it is the faster one for every M <= 16 (one pass
// over W, no per-weight work on the CUDA cores; whole-tile or cluster K-split
// schedules without global-memory round trips): on the 27B-class
// projections 16.0 / 16.7 / 21.6 us at M = 4 / 8 / 16 against 22.4 / 26.3 /
// ~35 us for the f16 tensor-core path.  The f16 path takes the shapes the
// FP4 path rejects (K % 256 != 0, K < 1024, N < 128, no workspace), the
// CUDA-core kernel what neither tensor-core path accepts.
DecodePath choose_path(int64_t M, int64_t N, int64_t K, bool workspace, const void *codes,
                       const void *scales) {
  if (M < 1 || M > kDecodeMaxM || N < 1 || K < 64 || K % 64) return DecodePath::kNone;
  const bool f4 = workspace && gemv_f4_supported(M, N, K, codes, scales);
  if (f4) return DecodePath::kFp4;
  const int tc_passes = gemv_tc_launches(M, N, K);
  if (tc_passes == 1) return DecodePath::kF16;
  if (tc_passes > 0) return DecodePath::kF16;
  return cuda_core_passes(M, N, K) ? DecodePath::kCudaCore : DecodePath::kNone;
}

}  // namespace

bool gemv_supported(int64_t M, int64_t N, int64_t K) {
  return choose_path(M, N, K, false, nullptr, nullptr) != DecodePath::kNone;
}

int gemv_launches(int64_t M, int64_t N, int64_t K, const char **kernel) {
  switch (choose_path(M, N, K, true, nullptr, nullptr)) {
    case DecodePath::kFp4:
      return gemv_f4_launches(M, N, K, kernel);
    case DecodePath::kF16:
      *kernel = "gemv_tc_kernel";
      return gemv_tc_launches(M, N, K);
    case DecodePath::kCudaCore:
      *kernel = "gemv_kernel";
      return cuda_core_passes(M, N, K);
    default:
      return 0;
  }
}

cudaError_t launch_gemv(const uint16_t *x, int64_t M, int64_t K, int64_t ldx, const uint8_t *codes,
                        const uint8_t *scales, const float *tensor_scale, int64_t N, uint16_t *y,
                        int64_t ldy, int32_t *status, void *workspace, cudaStream_t stream) {
  switch (choose_path(M, N, K, workspace != nullptr, codes, scales)) {
    case DecodePath::kFp4:
      return launch_gemv_f4(x, M, K, ldx, codes, scales, tensor_scale, N, y, ldy, status,
                            workspace, stream);
    case DecodePath::kF16:
      return launch_gemv_tc(x, M, K, ldx, codes, scales, tensor_scale, N, y, ldy, status, stream);
    case DecodePath::kCudaCore:
      break;
    default:
      return cudaErrorInvalidConfiguration;
  }
  for (int64_t m0 = 0; m0 < M;) {
    Plan p;
    const int MT = pass_tile(M - m0, N, K, p);
    if (MT == 0) return cudaErrorInvalidConfiguration;
    GemvArgs a;
    a.x = x + m0 * ldx;
    a.ldx = ldx;
    a.M = (int)((M - m0) < MT ? (M - m0) : MT);
    a.codes = codes;
    a.scales = scales;
    a.tensor_scale = tensor_scale;
    a.y = y + m0 * ldy;
    a.ldy = ldy;
    a.N = N;
    a.K = K;
    a.status = status;
    a.rows_per_stage = p.RS;
    a.nstages = p.NS;
    a.threads_per_row = p.P;
    a.row_groups = p.RG;
    a.scales_bulk = p.scales_bulk;
    a.stage_bytes = p.stage_bytes;
    a.codes_stage_bytes = p.codes_stage_bytes;
    int64_t grid = num_sms();
    if (grid > N) grid = N;
    const cudaError_t e = dispatch(a, p, (int)grid, stream);
    if (e != cudaSuccess) return e;
    m0 += MT;
  }
  return cudaSuccess;
}

}  // namespace impfp4
