// Shared device helpers for the NVFP4 kernels (sm_103a): mbarriers, bulk
// copies, bounded waits, element conversions through the Blackwell cvt
// instructions, and the device status word.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/imp_nvfp4.h"

namespace impfp4 {

// Every in-kernel wait gives up after this many nanoseconds of %globaltimer
// and reports IMP_DEV_TIMEOUT.  Kernels here run for micro- to milliseconds.
constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;  // 1 s

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void report(int32_t *status, int32_t flag) {
  if (status) atomicOr(status, flag);
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarrier ---------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("{\n.reg .b64 st;\nmbarrier.arrive.shared::cta.b64 st, [%0];\n}" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("{\n.reg .b64 st;\nmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of `bar` to complete.  Returns false (and reports
// IMP_DEV_TIMEOUT) if it has not after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, int32_t *status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      report(status, IMP_DEV_TIMEOUT);
      return false;
    }
  }
}

// ---- bulk copies (TMA, non-tensor form) --------------------------------------

// Copy `bytes` (multiple of 16, both addresses 16-byte aligned) from global
// to this CTA's shared memory; completion is signalled on `bar` as tx bytes.
__device__ __forceinline__ void bulk_g2s(void *smem_dst, const void *gmem_src, uint32_t bytes,
                                         uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// ---- element conversions -----------------------------------------------------

// Two E2M1 codes (one byte: element 2i low nibble, 2i+1 high nibble) -> f16x2
// (low half = element 2i).  Exact.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte_in_low_bits) {
  uint32_t out;
  asm("{\n.reg .b8 b0, b1, b2, b3;\nmov.b32 {b0, b1, b2, b3}, %1;\ncvt.rn.f16x2.e2m1x2 %0, b0;\n}"
      : "=r"(out)
      : "r"(byte_in_low_bits));
  return out;
}

// Four bytes of packed codes (8 elements) -> four f16x2 words, element order.
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n.reg .b8 b0, b1, b2, b3;\nmov.b32 {b0, b1, b2, b3}, %4;\n"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\ncvt.rn.f16x2.e2m1x2 %1, b1;\n"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\ncvt.rn.f16x2.e2m1x2 %3, b3;\n}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

// Two E4M3 bytes (low byte first) -> f16x2.  Exact for every finite E4M3 value.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
  uint32_t out;
  asm("{\n.reg .b16 lo;\nmov.b32 {lo, _}, %1;\ncvt.rn.f16x2.e4m3x2 %0, lo;\n}"
      : "=r"(out)
      : "r"(two_bytes));
  return out;
}

__device__ __forceinline__ float f16lo_to_f32(uint32_t h2) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu)));
}
__device__ __forceinline__ float f16hi_to_f32(uint32_t h2) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 >> 16)));
}

// Non-negative fp32 -> E4M3 byte: round to nearest even, saturating at 448
// (cvt .satfinite).  Both halves of the x2 result hold the same value.
__device__ __forceinline__ uint32_t f32_to_e4m3_satfinite(float u) {
  uint32_t out;
  asm("{\n.reg .b16 r;\ncvt.rn.satfinite.e4m3x2.f32 r, %1, %1;\ncvt.u32.u16 %0, r;\n}"
      : "=r"(out)
      : "f"(u));
  return out & 0xFFu;
}

// Eight fp32 values -> eight E2M1 codes (round to nearest even, saturating
// at 6, sign bit from the value), packed element 0 in the low nibble.
__device__ __forceinline__ uint32_t f32x8_to_e2m1_packed(const float (&q)[8]) {
  uint32_t out;
  asm("{\n.reg .b8 b0, b1, b2, b3;\n"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
      "mov.b32 %0, {b0, b1, b2, b3};\n}"
      : "=r"(out)
      : "f"(q[0]), "f"(q[1]), "f"(q[2]), "f"(q[3]), "f"(q[4]), "f"(q[5]), "f"(q[6]), "f"(q[7]));
  return out;
}

// fp32 accumulate of an f16 x f16 product: acc + a*b with a single rounding.
__device__ __forceinline__ float fma_f16f16_f32(uint16_t a, uint16_t b, float acc) {
  float d;
  asm("fma.rn.f32.f16 %0, %1, %2, %3;" : "=f"(d) : "h"(a), "h"(b), "f"(acc));
  return d;
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

__host__ __device__ inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// ---- split-tile hand-off (stream-K schedules) --------------------------------

// Launch epochs for the split-tile counters: consecutive from a random start
// per process (host).
unsigned long long next_launch_epoch();

// Counts one finished segment of a split tile; true for the tile's last.
// A counter is 16 bytes: the launch's epoch (64 bits), a check word derived
// from it (32 bits) and the count.  A value that does not carry this
// launch's epoch and check -- an earlier launch's, or whatever the workspace
// held before (a 2^-96 chance of a false match) -- counts as zero, so no
// call has to clear the counters; the last CTA of a tile still leaves zero,
// the first guess of the next launch.  Epochs start at a random value per
// process and grow by one per launch.
__device__ __forceinline__ bool count_split_segment(unsigned __int128 *c, unsigned long long epoch,
                                              int nslot) {
  const unsigned long long chk = (epoch * 0x9E3779B97F4A7C15ull) >> 32;
  unsigned __int128 old = 0;  // the tile's last CTA of each launch leaves zero
  while (true) {
    const unsigned long long hi = (unsigned long long)(old >> 64), lo = (unsigned long long)old;
    const unsigned long long cnt = (hi == epoch && (lo >> 32) == chk) ? (lo & 0xFFFFFFFFull) + 1 : 1;
    const unsigned __int128 nv = ((unsigned __int128)epoch << 64) | ((chk << 32) | cnt);
    const unsigned __int128 prev = atomicCAS(c, old, nv);
    if (prev == old) {
      if ((int)cnt != nslot) return false;
      __stcg(reinterpret_cast<uint4 *>(c), make_uint4(0, 0, 0, 0));  // for the next launch
      return true;
    }
    old = prev;  // not what was guessed: at most nslot + 1 rounds
  }
}


}  // namespace impfp4
