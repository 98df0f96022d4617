// NVFP4 quantizer (bf16 -> E2M1 codes + E4M3 block scales + fp32 tensor
// scale), bit-exact to the recipe in imp_nvfp4.h.
//
// Two HBM-bound passes over X:
//   1. amax_partial_kernel: one max|x| per CTA (as bf16 magnitude bits, which
//      order like the values; NaN/Inf bit patterns sort above every finite
//      value, so the same max detects them).
//   2. encode_kernel: every CTA folds the partial maxima into g and
//      s = g / 2688, then each thread encodes one 16-element block: block amax
//      a, u = (a/6)/s, E4M3 scale byte via cvt.rn.satfinite.e4m3x2, d = e4m3*s,
//      and 16 E2M1 codes via cvt.rn.satfinite.e2m1x2 on |x|/d with the sign
//      bit copied from x.  Every fp32 step is an explicitly rounded IEEE op
//      (__fdiv_rn, __fmul_rn), so no contraction or approximation can change
//      a byte.
#include <cuda.h>

#include <atomic>
#include <mutex>

#include "quantize.cuh"

namespace impfp4 {

namespace {

constexpr int kAmaxThreads = 256;
constexpr int64_t kAmaxSeg = 512;  // 16-byte vectors per amax segment (4096 elements)
constexpr int kEncThreads = 256;

__device__ __forceinline__ uint32_t warp_max_u32(uint32_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

// Per-half max of the magnitude bits of 8 bf16 values (sign bits cleared
// before comparing).
__device__ __forceinline__ uint32_t absmax8(uint4 a) {
  return __vmaxu2(__vmaxu2(a.x & 0x7FFF7FFFu, a.y & 0x7FFF7FFFu),
                  __vmaxu2(a.z & 0x7FFF7FFFu, a.w & 0x7FFF7FFFu));
}

// Block-wide max of a per-thread value; result valid in every thread.
template <int kThreads>
__device__ __forceinline__ uint32_t block_max_u32(uint32_t v, uint32_t *red) {
  v = warp_max_u32(v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  uint32_t r = (lane < kThreads / 32) ? red[lane] : 0u;
  r = warp_max_u32(r);
  __syncthreads();
  return r;
}

// Pass 1: per-CTA max of |x| as bf16 magnitude bits.  Warps stride over
// segments of kAmaxSeg 16-byte vectors (4096 elements) of a row, so that a
// tensor of few long rows (an activation) still spreads over every SM;
// lanes read four vectors at a time.
__global__ void __launch_bounds__(kAmaxThreads) amax_partial_kernel(const uint16_t *__restrict__ x,
                                                                    int64_t rows, int64_t K,
                                                                    int64_t ldx,
                                                                    uint32_t *__restrict__ partial,
                                                                    int32_t *status) {
  // the encode pass may be launched now; it waits for this grid to finish
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ uint32_t red[kAmaxThreads / 32];
  const int lane = threadIdx.x & 31;
  const int64_t warps_total = (int64_t)gridDim.x * (kAmaxThreads / 32);
  const int64_t vec_per_row = K / 8;
  const int64_t nseg = ceil_div(vec_per_row, kAmaxSeg);
  uint32_t m2 = 0;  // two 16-bit maxima side by side
  for (int64_t g = (int64_t)blockIdx.x * (kAmaxThreads / 32) + (threadIdx.x >> 5); g < rows * nseg;
       g += warps_total) {
    const int64_t r = g / nseg, v0 = (g - r * nseg) * kAmaxSeg;
    const int64_t v1 = v0 + kAmaxSeg < vec_per_row ? v0 + kAmaxSeg : vec_per_row;
    const uint4 *row = reinterpret_cast<const uint4 *>(x + r * ldx);
    int64_t v = v0 + lane;
    for (; v + 96 < v1; v += 128) {
      const uint4 a = __ldg(row + v), b = __ldg(row + v + 32), c = __ldg(row + v + 64),
                  d = __ldg(row + v + 96);
      m2 = __vmaxu2(m2, __vmaxu2(__vmaxu2(absmax8(a), absmax8(b)), __vmaxu2(absmax8(c), absmax8(d))));
    }
    for (; v < v1; v += 32) m2 = __vmaxu2(m2, absmax8(__ldg(row + v)));
  }
  uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
  m = block_max_u32<kAmaxThreads>(m, red);
  if (threadIdx.x == 0) {
    partial[blockIdx.x] = m;
    if (m >= 0x7F80u) report(status, IMP_DEV_NONFINITE_INPUT);
  }
}

// The codes of q_i = RN(x_i / d) for eight elements (signed; the E2M1
// conversion keeps the sign, also of a zero) without eight IEEE divisions.
// x_i * RN(1/d) is within 2^-22.4 (relative) of RN(x_i / d); the products
// with RN(1/d) (1 -/+ 2^-20) therefore bracket RN(x_i / d) in magnitude, and
// rounding to E2M1 is monotone in the magnitude: if both brackets give the
// same codes, those are the codes of the quotients.  Only when an element
// sits that close to a rounding boundary (or 1/d is not finite) are the
// eight quotients divided exactly.
__device__ __forceinline__ uint32_t e2m1x8_of_quotients(const float (&x)[8], float d, float inv_lo,
                                                        float inv_hi) {
  float lo[8], hi[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    lo[i] = __fmul_rn(x[i], inv_lo);
    hi[i] = __fmul_rn(x[i], inv_hi);
  }
  const uint32_t c = f32x8_to_e2m1_packed(lo);
  if (c == f32x8_to_e2m1_packed(hi) && inv_hi < INFINITY) return c;
  float q[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) q[i] = __fdiv_rn(x[i], d);
  return f32x8_to_e2m1_packed(q);
}

// The E4M3 block scale of u = RN(RN(a / 6) / s) the same way: a times
// RN(RN(1/6) RN(1/s)) is within 2^-21.7 of u; bracketed by (1 -/+ 2^-20),
// the exact two divisions run only next to a rounding boundary.
__device__ __forceinline__ uint32_t e4m3_block_scale(float a, float s, float c_lo, float c_hi) {
  if (s == 0.0f) return 0u;
  const uint32_t lo = f32_to_e4m3_satfinite(__fmul_rn(a, c_lo));
  if (lo == f32_to_e4m3_satfinite(__fmul_rn(a, c_hi)) && c_hi < INFINITY) return lo;
  return f32_to_e4m3_satfinite(__fdiv_rn(__fdiv_rn(a, 6.0f), s));
}

// Pass 2: fold the partial maxima, then encode one 16-element block per thread.
// MMA_LAYOUT: write the scale bytes in the tensor-core atom layout
// (mma_scale_offset) instead of row-major.
template <bool MMA_LAYOUT>
__global__ void __launch_bounds__(kEncThreads) encode_kernel(
    const uint16_t *__restrict__ x, int64_t rows, int64_t K, int64_t ldx,
    const uint32_t *__restrict__ partial, int num_partial, uint8_t *__restrict__ codes,
    uint8_t *__restrict__ scales, float *__restrict__ tensor_scale) {
  __shared__ uint32_t red[kEncThreads / 32];
  // Launched early after the amax pass (programmatic dependent launch): the
  // GEMM that reads the codes may be launched in turn, and nothing is read
  // before the amax pass has finished and its partial maxima are visible.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  uint32_t m = 0;
  for (int i = threadIdx.x; i < num_partial; i += kEncThreads) m = max(m, partial[i]);
  m = block_max_u32<kEncThreads>(m, red);
  const float g = bf16_bits_to_f32(m < 0x7F80u ? m : 0u);
  const float s = __fdiv_rn(g, 2688.0f);
  if (blockIdx.x == 0 && threadIdx.x == 0) *tensor_scale = s;
  constexpr float kDown = 1.0f - 0x1p-20f, kUp = 1.0f + 0x1p-20f;
  const float c6s = __fmul_rn(__frcp_rn(6.0f), __frcp_rn(s));  // ~ 1 / (6 s)
  const float c_lo = __fmul_rn(c6s, kDown), c_hi = __fmul_rn(c6s, kUp);

  // Warps stride over segments of 64 consecutive blocks of a row; each lane
  // encodes blocks lane and lane + 32 of its warp's segment, both loaded
  // before either is encoded (four 16-byte loads in flight per thread).
  const int64_t blocks_per_row = K / 16;
  const int64_t segs_per_row = ceil_div(blocks_per_row, 64);
  const int64_t total_segs = rows * segs_per_row;
  const int lane = threadIdx.x & 31;
  // (32-bit index arithmetic while the segment count allows: a 64-bit
  // division per segment costs more than the block's encoding)
  const bool narrow = total_segs < (int64_t)0x7FFFFFFF;
  const uint32_t spr32 = (uint32_t)segs_per_row;
  auto encode = [&](const uint4 v0, const uint4 v1, int64_t r, int64_t b) {
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    uint32_t a2 = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) a2 = __vmaxu2(a2, w[i] & 0x7FFF7FFFu);
    const float a = bf16_bits_to_f32(max(a2 & 0xFFFFu, a2 >> 16));
    const uint32_t sb = e4m3_block_scale(a, s, c_lo, c_hi);
    const float d = __fmul_rn(f16lo_to_f32(e4m3x2_to_f16x2(sb)), s);
    uint32_t packed[2] = {0u, 0u};
    if (d != 0.0f) {
      const float inv = __frcp_rn(d);
      const float inv_lo = __fmul_rn(inv, kDown), inv_hi = __fmul_rn(inv, kUp);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float xv[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t wi = w[4 * h + i];
          xv[2 * i] = bf16_bits_to_f32(wi & 0xFFFFu);
          xv[2 * i + 1] = bf16_bits_to_f32(wi >> 16);
        }
        packed[h] = e2m1x8_of_quotients(xv, d, inv_lo, inv_hi);
      }
    }
    *reinterpret_cast<uint2 *>(codes + r * (K / 2) + b * 8) = make_uint2(packed[0], packed[1]);
    if (MMA_LAYOUT)
      scales[mma_scale_offset(r, b, K)] = static_cast<uint8_t>(sb);
    else
      scales[r * blocks_per_row + b] = static_cast<uint8_t>(sb);
  };
  for (int64_t seg = (int64_t)blockIdx.x * (kEncThreads / 32) + (threadIdx.x >> 5); seg < total_segs;
       seg += (int64_t)gridDim.x * (kEncThreads / 32)) {
    int64_t r, b;
    if (narrow) {
      const uint32_t r32 = (uint32_t)seg / spr32;
      r = r32;
      b = (int64_t)(((uint32_t)seg - r32 * spr32) * 64u + (uint32_t)lane);
    } else {
      r = seg / segs_per_row;
      b = (seg - r * segs_per_row) * 64 + lane;
    }
    if (b >= blocks_per_row) continue;
    const uint4 *src = reinterpret_cast<const uint4 *>(x + r * ldx + b * 16);
    const bool two = b + 32 < blocks_per_row;
    const uint4 v0 = __ldg(src), v1 = __ldg(src + 1);
    uint4 v2 = make_uint4(0, 0, 0, 0), v3 = v2;
    if (two) {
      v2 = __ldg(src + 64);  // block b + 32: 32 blocks x 32 bytes further
      v3 = __ldg(src + 65);
    }
    encode(v0, v1, r, b);
    if (two) encode(v2, v3, r, b + 32);
  }
}

// SM count of the current device, cached per device (threads may race to
// fill an entry: they store the same value).
int num_sms_cached() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

// One warp per row at a time; at most kMaxPartials CTAs, so the workspace
// size does not depend on the device.
constexpr int kMaxPartials = 1024;

int amax_grid(int64_t rows, int64_t K) {
  int64_t g = ceil_div(rows * ceil_div(K / 8, kAmaxSeg), kAmaxThreads / 32);
  if (g > kMaxPartials) g = kMaxPartials;
  if (g < 1) g = 1;
  return static_cast<int>(g);
}

}  // namespace

int num_sms() { return num_sms_cached(); }

size_t quantize_workspace_bytes(int64_t rows, int64_t K) {
  return static_cast<size_t>(amax_grid(rows, K)) * sizeof(uint32_t);
}

cudaError_t launch_quantize(const uint16_t *x, int64_t rows, int64_t K, int64_t ldx,
                            uint8_t *codes, uint8_t *scales, float *tensor_scale,
                            int32_t *status, void *workspace, cudaStream_t stream) {
  const int ga = amax_grid(rows, K);
  uint32_t *partial = static_cast<uint32_t *>(workspace);
  amax_partial_kernel<<<ga, kAmaxThreads, 0, stream>>>(x, rows, K, ldx, partial, status);
  const int64_t segs = rows * ceil_div(K / 16, 64);
  int64_t ge = ceil_div(segs, kEncThreads / 32);
  const int64_t cap = (int64_t)num_sms_cached() * 8;
  if (ge > cap) ge = cap;
  if (ge < 1) ge = 1;
  encode_kernel<false><<<static_cast<int>(ge), kEncThreads, 0, stream>>>(
      x, rows, K, ldx, partial, ga, codes, scales, tensor_scale);
  return cudaGetLastError();
}

namespace {

// One thread per 4-byte word of the atom layout: word w of atom (rb, kc)
// holds row rb*128 + 32*(w % 4) + w / 4, blocks 4*kc .. 4*kc+3.
__global__ void scale_relayout_kernel(const uint8_t *__restrict__ scales, int64_t rows, int64_t K,
                                      uint8_t *__restrict__ mma_scales, int64_t total_words) {
  const int64_t KB = K / 16, KA = K / 64;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total_words;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t atom = i / 128, w = i % 128;
    const int64_t rb = atom / KA, kc = atom % KA;
    const int64_t r = rb * 128 + 32 * (w % 4) + w / 4;
    uint32_t v = 0;
    if (r < rows) v = *reinterpret_cast<const uint32_t *>(scales + r * KB + 4 * kc);
    reinterpret_cast<uint32_t *>(mma_scales)[i] = v;
  }
}

// One thread per 16-byte unit of the tile layout.
__global__ void code_relayout_kernel(const uint8_t *__restrict__ codes, int64_t rows, int64_t K,
                                     uint8_t *__restrict__ mma_codes, int64_t total_units) {
  const int64_t KH = K / 2, nch = mma_code_chunks(K);
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total_units;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t tile = i / 1024, w = i % 1024;  // 1024 units of 16 B per tile
    const int64_t rb = tile / nch, c = tile % nch;
    const int rr = (int)(w / 8), up = (int)(w % 8);   // row in tile, stored unit
    const int u = up ^ (rr & 7);                       // logical unit of that row
    const int64_t r = rb * 128 + rr, kb = c * 128 + 16 * u;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r < rows && kb < KH) v = *reinterpret_cast<const uint4 *>(codes + r * KH + kb);
    reinterpret_cast<uint4 *>(mma_codes)[i] = v;
  }
}

}  // namespace

cudaError_t launch_code_relayout(const uint8_t *codes, int64_t rows, int64_t K, uint8_t *mma_codes,
                                 cudaStream_t stream) {
  const int64_t units = (int64_t)mma_code_bytes(rows, K) / 16;
  int64_t grid = ceil_div(units, 256);
  const int64_t cap = (int64_t)num_sms_cached() * 8;
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  code_relayout_kernel<<<(int)grid, 256, 0, stream>>>(codes, rows, K, mma_codes, units);
  return cudaGetLastError();
}

cudaError_t launch_scale_relayout(const uint8_t *scales, int64_t rows, int64_t K,
                                  uint8_t *mma_scales, cudaStream_t stream) {
  const int64_t words = (int64_t)mma_scale_bytes(rows, K) / 4;
  int64_t grid = ceil_div(words, 256);
  const int64_t cap = (int64_t)num_sms_cached() * 8;
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  scale_relayout_kernel<<<(int)grid, 256, 0, stream>>>(scales, rows, K, mma_scales, words);
  return cudaGetLastError();
}

// ---- allocation-free variant -------------------------------------------------
//
// Scratch of imp_nvfp4_quantize_noalloc: the per-CTA partial maxima of pass
// 1, in a fixed device array instead of caller-provided workspace.  Every
// GPU that loads the library holds these 4 KB until the process exits.
namespace {
__device__ __align__(256) uint32_t g_noalloc_partials[kMaxPartials];
}

size_t quantize_noalloc_capacity() { return sizeof(g_noalloc_partials); }

namespace {

// ID of the calling thread's current CUDA context (0 if none or unknown),
// through the driver's cuCtxGetCurrent / cuCtxGetId, looked up once.
unsigned long long current_context_id() {
  using GetCurrent = CUresult (*)(CUcontext *);
  using GetId = CUresult (*)(CUcontext, unsigned long long *);
  static const GetCurrent get_current = []() {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      fn = nullptr;
    return reinterpret_cast<GetCurrent>(fn);
  }();
  static const GetId get_id = []() {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      fn = nullptr;
    return reinterpret_cast<GetId>(fn);
  }();
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// The device address of g_noalloc_partials, per device, for the context it
// was looked up in: a device reset or a new primary context loads the module
// again (a new address), so a cached address is used only while the current
// context is the one it came from.  One mutex per device guards the entry.
struct NoallocAddr {
  std::mutex mu;
  unsigned long long ctx = 0;
  void *addr = nullptr;
};
NoallocAddr g_noalloc_addr[64];

}  // namespace

cudaError_t launch_quantize_noalloc(const uint16_t *x, int64_t rows, int64_t K, int64_t ldx,
                                    uint8_t *codes, uint8_t *scales, float *tensor_scale,
                                    int32_t *status, cudaStream_t stream) {
  if (quantize_workspace_bytes(rows, K) > sizeof(g_noalloc_partials))
    return cudaErrorInvalidValue;  // caller checks sizes first; kept as a guard
  // In host code g_noalloc_partials names a host-side shadow, not device
  // memory: the device address is looked up with the device current.
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  NoallocAddr &slot = g_noalloc_addr[dev];
  void *addr = nullptr;
  {
    std::lock_guard<std::mutex> lock(slot.mu);
    const unsigned long long ctx = current_context_id();
    if (ctx != 0 && ctx == slot.ctx && slot.addr) {
      addr = slot.addr;
    } else {
      e = cudaGetSymbolAddress(&addr, g_noalloc_partials);
      if (e != cudaSuccess) return e;
      // the lookup makes the device's context current if it was not yet
      slot.ctx = ctx != 0 ? ctx : current_context_id();
      slot.addr = addr;
    }
  }
  // Pass 1 writes every partial that pass 2 reads, so the array needs no
  // clearing between calls.
  return launch_quantize(x, rows, K, ldx, codes, scales, tensor_scale, status, addr, stream);
}

cudaError_t launch_encode_with_amax(const uint16_t *x, int64_t rows, int64_t K, int64_t ldx,
                                   const uint32_t *amax_bits, uint8_t *codes, uint8_t *scales,
                                   float *tensor_scale, bool mma_layout, cudaStream_t stream) {
  const int64_t segs = rows * ceil_div(K / 16, 64);
  int64_t ge = ceil_div(segs, kEncThreads / 32);
  const int64_t cap = (int64_t)num_sms_cached() * 8;
  if (ge > cap) ge = cap;
  if (ge < 1) ge = 1;
  if (mma_layout)
    encode_kernel<true><<<static_cast<int>(ge), kEncThreads, 0, stream>>>(
        x, rows, K, ldx, amax_bits, 1, codes, scales, tensor_scale);
  else
    encode_kernel<false><<<static_cast<int>(ge), kEncThreads, 0, stream>>>(
        x, rows, K, ldx, amax_bits, 1, codes, scales, tensor_scale);
  return cudaGetLastError();
}

cudaError_t launch_quantize_mma(const uint16_t *x, int64_t rows, int64_t K, int64_t ldx,
                                uint8_t *codes, uint8_t *mma_scales, float *tensor_scale,
                                int32_t *status, void *workspace, cudaStream_t stream) {
  const int ga = amax_grid(rows, K);
  uint32_t *partial = static_cast<uint32_t *>(workspace);
  amax_partial_kernel<<<ga, kAmaxThreads, 0, stream>>>(x, rows, K, ldx, partial, status);
  const int64_t segs = rows * ceil_div(K / 16, 64);
  int64_t ge = ceil_div(segs, kEncThreads / 32);
  const int64_t cap = (int64_t)num_sms_cached() * 8;
  if (ge > cap) ge = cap;
  if (ge < 1) ge = 1;
  // the encode pass with programmatic dependent launch (it waits in-kernel)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ge);
  cfg.blockDim = dim3(kEncThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, encode_kernel<true>, x, rows, K, ldx,
                                           static_cast<const uint32_t *>(partial), ga, codes,
                                           mma_scales, tensor_scale);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// ---- MXFP4 (OCP MX v1.0) and FP8-E4M3 weights ---------------------------------
//
// MXFP4: 32-element blocks along K, one E8M0 scale byte (2^(b - 127)) per
// block, E2M1 codes.  Shared exponent e = floor(log2(block amax)) - 2,
// clamped to [-127, 127]; code = E2M1(|x| * 2^-e), nearest even, saturating
// at 6 (cvt.rn.satfinite.e2m1x2), sign bit copied from x.  Multiplying by the
// power of two 2^-e is exact (it is a normal float for every e a bf16 block
// can give), so the codes equal those of the division x / 2^e.
//
// FP8 weights: one fp32 scale s8 = g / 448 per tensor (the global amax pass
// of the NVFP4 quantizer), code = E4M3(|x| / s8) (cvt.rn.satfinite.e4m3x2),
// sign bit copied from x; s8 == 0 gives all codes 0.
namespace {

constexpr int kMxThreads = 256;

// floor(log2 v) of a nonzero finite bf16 magnitude (bits without the sign).
__device__ __forceinline__ int bf16_floor_log2(uint32_t mag) {
  const int E = (int)(mag >> 7);
  if (E > 0) return E - 127;
  return (31 - __clz((int)mag)) - 133;  // subnormal: mantissa * 2^-133
}

// One thread per 32-element block.
__global__ void __launch_bounds__(kMxThreads) mx_quantize_kernel(
    const uint16_t *__restrict__ x, int64_t rows, int64_t K, int64_t ldx,
    uint8_t *__restrict__ codes, uint8_t *__restrict__ scales, int32_t *status) {
  const int64_t nb = K / 32, total = rows * nb;
  for (int64_t i = (int64_t)blockIdx.x * kMxThreads + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * kMxThreads) {
    const int64_t r = i / nb, b = i - r * nb;
    const uint4 *src = reinterpret_cast<const uint4 *>(x + r * ldx + 32 * b);
    uint32_t w[16];
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const uint4 t = __ldg(src + v);
      w[4 * v] = t.x;
      w[4 * v + 1] = t.y;
      w[4 * v + 2] = t.z;
      w[4 * v + 3] = t.w;
    }
    uint32_t a2 = 0;
#pragma unroll
    for (int v = 0; v < 16; ++v) a2 = __vmaxu2(a2, w[v] & 0x7FFF7FFFu);
    const uint32_t amag = max(a2 & 0xFFFFu, a2 >> 16);
    if (amag >= 0x7F80u) report(status, IMP_DEV_NONFINITE_INPUT);
    int e = amag ? bf16_floor_log2(amag) - 2 : -127;
    e = min(127, max(-127, e));
    scales[r * nb + b] = (uint8_t)(e + 127);
    const float inv = __uint_as_float((uint32_t)(127 - e) << 23);  // 2^-e, e <= 126 here
    uint32_t packed[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      float q[8];
      uint32_t sign = 0;
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const uint32_t wi = w[4 * h + v];
        q[2 * v] = __fmul_rn(bf16_bits_to_f32(wi & 0x7FFFu), inv);
        q[2 * v + 1] = __fmul_rn(bf16_bits_to_f32((wi >> 16) & 0x7FFFu), inv);
        sign |= ((wi >> 15) & 1u) << (8 * v + 3);
        sign |= (wi >> 31) << (8 * v + 7);
      }
      packed[h] = f32x8_to_e2m1_packed(q) | sign;
    }
    *reinterpret_cast<uint4 *>(codes + r * (K / 2) + 16 * b) =
        make_uint4(packed[0], packed[1], packed[2], packed[3]);
  }
}

// Two E4M3 bytes (element 0 in the low byte) of two non-negative floats.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
  uint32_t out;
  asm("{\n.reg .b16 r;\ncvt.rn.satfinite.e4m3x2.f32 r, %2, %1;\ncvt.u32.u16 %0, r;\n}"
      : "=r"(out)
      : "f"(lo), "f"(hi));
  return out;
}

// FP8 pass 2: s8 from the partial maxima, then one thread per 8 elements.
__global__ void __launch_bounds__(kEncThreads) fp8_encode_kernel(
    const uint16_t *__restrict__ x, int64_t rows, int64_t K, int64_t ldx,
    const uint32_t *__restrict__ partial, int num_partial, uint8_t *__restrict__ codes,
    float *__restrict__ tensor_scale) {
  __shared__ uint32_t red[kEncThreads / 32];
  uint32_t m = 0;
  for (int i = threadIdx.x; i < num_partial; i += kEncThreads) m = max(m, partial[i]);
  m = block_max_u32<kEncThreads>(m, red);
  const float g = bf16_bits_to_f32(m < 0x7F80u ? m : 0u);
  const float s8 = __fdiv_rn(g, 448.0f);
  const float inv8 = __frcp_rn(s8);
  if (blockIdx.x == 0 && threadIdx.x == 0) *tensor_scale = s8;
  const int64_t per_row = K / 8, total = rows * per_row;
  for (int64_t i = (int64_t)blockIdx.x * kEncThreads + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * kEncThreads) {
    const int64_t r = i / per_row, j = i - r * per_row;
    uint2 out = make_uint2(0u, 0u);
    if (s8 != 0.0f) {
      const uint4 t = __ldg(reinterpret_cast<const uint4 *>(x + r * ldx + 8 * j));
      const uint32_t w[4] = {t.x, t.y, t.z, t.w};
      float m[8];
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        m[2 * v] = bf16_bits_to_f32(w[v] & 0x7FFFu);
        m[2 * v + 1] = bf16_bits_to_f32((w[v] >> 16) & 0x7FFFu);
      }
      // as e2m1x8_of_quotients: m * RN(1/s8), with the exact division only
      // next to a rounding boundary of E4M3
      constexpr float kDown = 1.0f - 0x1p-20f, kUp = 1.0f + 0x1p-20f;
      uint32_t b[4];
      bool exact = true;
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const float q0 = __fmul_rn(m[2 * v], inv8), q1 = __fmul_rn(m[2 * v + 1], inv8);
        b[v] = f32x2_to_e4m3x2(q0, q1);
        exact = exact && b[v] == f32x2_to_e4m3x2(__fmul_rn(q0, kDown), __fmul_rn(q1, kDown)) &&
                b[v] == f32x2_to_e4m3x2(__fmul_rn(q0, kUp), __fmul_rn(q1, kUp));
      }
      if (!exact || !(inv8 < INFINITY)) {
#pragma unroll
        for (int v = 0; v < 4; ++v)
          b[v] = f32x2_to_e4m3x2(__fdiv_rn(m[2 * v], s8), __fdiv_rn(m[2 * v + 1], s8));
      }
#pragma unroll
      for (int v = 0; v < 4; ++v) b[v] |= ((w[v] >> 8) & 0x80u) | ((w[v] >> 16) & 0x8000u);
      out = make_uint2(b[0] | b[1] << 16, b[2] | b[3] << 16);
    }
    *reinterpret_cast<uint2 *>(codes + r * K + 8 * j) = out;
  }
}

// MXFP4 -> NVFP4, pass 1: the largest E8M0 byte among 16-element halves of a
// block that hold a nonzero code (atomicMax into *bmax, zeroed beforehand).
__global__ void __launch_bounds__(256) mx_scale_max_kernel(const uint8_t *__restrict__ codes,
                                                           const uint8_t *__restrict__ scales,
                                                           int64_t halves, uint32_t *bmax) {
  __shared__ uint32_t red[8];
  uint32_t m = 0;
  for (int64_t h = (int64_t)blockIdx.x * 256 + threadIdx.x; h < halves;
       h += (int64_t)gridDim.x * 256) {
    const uint2 c = *reinterpret_cast<const uint2 *>(codes + 8 * h);
    if ((c.x | c.y) & 0x77777777u) m = max(m, (uint32_t)scales[h / 2]);
  }
  m = block_max_u32<256>(m, red);
  if (threadIdx.x == 0 && m) atomicMax(bmax, m);
}

// E4M3 byte of 2^k for k in [-9, 8] (normal from 2^-6, subnormal below).
__device__ __forceinline__ uint32_t e4m3_pow2(int k) {
  return k >= -6 ? (uint32_t)(k + 7) << 3 : 1u << (k + 9);
}

// Pass 2: each half gets the E4M3 scale 2^(b - bmax + 8), exact while that
// is at least 2^-9; a half whose codes are all zero gets 0x00; a half with
// nonzero codes more than 2^17 below the largest is reported
// (IMP_DEV_RANGE).  Block 0 writes the tensor scale 2^(bmax - 135).
__global__ void __launch_bounds__(256) mx_to_nvfp4_kernel(
    const uint8_t *__restrict__ codes, const uint8_t *__restrict__ scales, int64_t halves,
    const uint32_t *__restrict__ bmax_p, uint8_t *__restrict__ nv_scales, float *tensor_scale,
    int32_t *status) {
  const int bmax = (int)*bmax_p;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    const int t = bmax - 135;  // exponent of the tensor scale, in [-135, 119]
    *tensor_scale = t >= -126 ? __uint_as_float((uint32_t)(t + 127) << 23)
                              : __uint_as_float(1u << (t + 149));
  }
  for (int64_t h = (int64_t)blockIdx.x * 256 + threadIdx.x; h < halves;
       h += (int64_t)gridDim.x * 256) {
    const uint2 c = *reinterpret_cast<const uint2 *>(codes + 8 * h);
    uint32_t out = 0;
    if ((c.x | c.y) & 0x77777777u) {
      const int k = (int)scales[h / 2] - bmax + 8;
      if (k < -9) report(status, IMP_DEV_RANGE);
      else out = e4m3_pow2(k);
    }
    nv_scales[h] = (uint8_t)out;
  }
}

int grid_for(int64_t items, int threads) {
  int64_t g = ceil_div(items, threads);
  const int64_t cap = (int64_t)num_sms_cached() * 8;
  if (g > cap) g = cap;
  if (g < 1) g = 1;
  return (int)g;
}

}  // namespace

cudaError_t launch_mx_quantize(const uint16_t *x, int64_t rows, int64_t K, int64_t ldx,
                               uint8_t *codes, uint8_t *scales, int32_t *status,
                               cudaStream_t stream) {
  mx_quantize_kernel<<<grid_for(rows * (K / 32), kMxThreads), kMxThreads, 0, stream>>>(
      x, rows, K, ldx, codes, scales, status);
  return cudaGetLastError();
}

cudaError_t launch_fp8_quantize(const uint16_t *x, int64_t rows, int64_t K, int64_t ldx,
                                uint8_t *codes, float *tensor_scale, int32_t *status,
                                void *workspace, cudaStream_t stream) {
  const int ga = amax_grid(rows, K);
  uint32_t *partial = static_cast<uint32_t *>(workspace);
  amax_partial_kernel<<<ga, kAmaxThreads, 0, stream>>>(x, rows, K, ldx, partial, status);
  fp8_encode_kernel<<<grid_for(rows * (K / 8), kEncThreads), kEncThreads, 0, stream>>>(
      x, rows, K, ldx, partial, ga, codes, tensor_scale);
  return cudaGetLastError();
}

cudaError_t launch_mx_to_nvfp4(const uint8_t *codes, const uint8_t *mx_scales, int64_t rows,
                               int64_t K, uint8_t *out_codes, uint8_t *nv_scales,
                               float *tensor_scale, int32_t *status, void *workspace,
                               cudaStream_t stream) {
  uint32_t *bmax = static_cast<uint32_t *>(workspace);
  const int64_t halves = rows * (K / 16);
  cudaError_t e = cudaMemsetAsync(bmax, 0, sizeof(uint32_t), stream);
  if (e != cudaSuccess) return e;
  if (out_codes != codes) {
    e = cudaMemcpyAsync(out_codes, codes, (size_t)rows * (size_t)(K / 2), cudaMemcpyDeviceToDevice,
                        stream);
    if (e != cudaSuccess) return e;
  }
  mx_scale_max_kernel<<<grid_for(halves, 256), 256, 0, stream>>>(codes, mx_scales, halves, bmax);
  mx_to_nvfp4_kernel<<<grid_for(halves, 256), 256, 0, stream>>>(codes, mx_scales, halves, bmax,
                                                                nv_scales, tensor_scale, status);
  return cudaGetLastError();
}

}  // namespace impfp4
