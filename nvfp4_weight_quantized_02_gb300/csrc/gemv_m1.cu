// Decode GEMV at M = 1: y[n] = s * sum_k x[k] * e2m1(c[n][k]) * e4m3(sb[n][k/16]).
//
// Decode is bandwidth-bound (imp README, "How it works"; "1. The big
// picture", section "The most important number in this book"), so the kernel
// is shaped to stream W at HBM speed with as few instructions per weight as
// possible:
//
//  * Persistent grid, one CTA per SM; CTA c owns rows [N*c/G, N*(c+1)/G).
//  * A producer thread streams stages of RS whole rows (codes, and scales when
//    K % 256 == 0) into a shared-memory ring with 1-D bulk copies
//    (cp.async.bulk + mbarrier transaction counts); rows of the [N][K/2] code
//    array are contiguous, so a stage is one copy per array.
//  * The multiply-accumulate runs on the tensor cores (mma.sync m16n8k16,
//    f16 x f16 -> f32).  For one "unit" of two rows x 1024 k:
//      lane L (= 4g + t) owns the two 16-element blocks 2L and 2L+1 of the
//      unit in both rows: one 16-byte shared-memory read per row, all 32
//      lanes reading 512 contiguous bytes (no bank conflicts).
//      A row g    = row n,   the block group of lanes 4g..4g+3,
//      A row g+8  = row n+1, the same block group,
//      B column g = X at that block group's k,
//    so D[g][g] and D[g+8][g] are the two rows' partial dot products over
//    block group g; the other D entries are never read.  Eight mma steps
//    cover the unit (step s takes elements 4(s%4)..4(s%4)+3 of block
//    2L + s/4 in every lane).
//  * A fragments: cvt.rn.f16x2.e2m1x2 per code byte, multiplied (HMUL2) by
//    the block's E4M3 scale (cvt.rn.f16x2.e4m3x2).  e2m1 * e4m3 has at most
//    6 significant bits and lies in [2^-10, 2688], so it is exact in f16.
//  * B fragments: each warp owns a fixed K-slice and keeps X for it in
//    registers as f16, scaled by one power of two 2^sh per call so that
//    max|x| lies in [2^14, 2^15): exact for every element within 2^24 of the
//    largest (smaller ones round to f16 subnormals: an absolute error below
//    max|x| * 2^-39 per element).  The factor is undone in fp32 at the end.
//  * Products are exact; sums are fp32 (tensor-core accumulation across the
//    warp's units, then a shuffle butterfly, then a fixed-order sum of the
//    per-warp partials), times the tensor scale, rounded to bf16.  No step
//    depends on timing, so results are bitwise reproducible.
#include "gemv.cuh"

namespace impfp4 {

namespace {

constexpr int kProducer = 32;
constexpr int kMaxStages = 8;
constexpr size_t kSmemBudget = 200 * 1024;
constexpr size_t kHeadBytes = 2 * kMaxStages * sizeof(uint64_t) + 16;
constexpr int kUnitK = 1024;  // k per unit (per warp step over two rows)

struct M1Args {
  const uint16_t *x;
  const uint8_t *codes;
  const uint8_t *scales;
  const float *tensor_scale;
  uint16_t *y;
  int64_t N, K;
  int32_t *status;
  int rows_per_stage;  // RS (even)
  int nstages;         // NS
  int warps_per_row;   // NWK: warps splitting K
  int row_groups;      // RG: groups of warps taking different row pairs
  int rows_per_block;  // RB: rows whose partial sums are reduced together
  int scales_bulk;
  uint32_t stage_bytes, codes_stage_bytes;
};

__device__ __forceinline__ void named_bar(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ __half2 u32_as_h2(uint32_t v) { return *reinterpret_cast<__half2 *>(&v); }
__device__ __forceinline__ uint32_t h2_as_u32(__half2 v) { return *reinterpret_cast<uint32_t *>(&v); }

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t f16x2_pack(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&h);
}

// One unit: rows (n, n+1), 1024 k.  cw0/cw1: the lane's 16 code bytes of
// each row; sc0/sc1: its two scale bytes of each row; xr: the lane's 32 X
// values as 16 f16x2.  d and e are two independent accumulator chains.
__device__ __forceinline__ void unit_mma(float (&d)[4], float (&e)[4], const uint4 cw0,
                                         const uint4 cw1, uint32_t sc0, uint32_t sc1,
                                         const uint32_t (&xr)[16]) {
  const __half2 s0 = u32_as_h2(e4m3x2_to_f16x2(sc0));  // (block 2L, block 2L+1) of row n
  const __half2 s1 = u32_as_h2(e4m3x2_to_f16x2(sc1));  // same blocks of row n+1
  const uint32_t w0[4] = {cw0.x, cw0.y, cw0.z, cw0.w};
  const uint32_t w1[4] = {cw1.x, cw1.y, cw1.z, cw1.w};
#pragma unroll
  for (int blk = 0; blk < 2; ++blk) {
    const __half2 sa = blk ? __high2half2(s0) : __low2half2(s0);  // block scale, both halves
    const __half2 sb = blk ? __high2half2(s1) : __low2half2(s1);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      uint32_t h0[4], h1[4];  // 4 bytes = 8 elements = two mma steps
      e2m1x8_to_f16x2x4(w0[2 * blk + half], h0);
      e2m1x8_to_f16x2x4(w1[2 * blk + half], h1);
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int ei = 8 * blk + 4 * half + 2 * q;  // f16x2 index of elements 4s'..4s'+1
        mma16816(q ? e : d, h2_as_u32(__hmul2(u32_as_h2(h0[2 * q]), sa)),
                 h2_as_u32(__hmul2(u32_as_h2(h1[2 * q]), sb)),
                 h2_as_u32(__hmul2(u32_as_h2(h0[2 * q + 1]), sa)),
                 h2_as_u32(__hmul2(u32_as_h2(h1[2 * q + 1]), sb)), xr[ei], xr[ei + 1]);
      }
    }
  }
}

// Consumer warps per CTA an instantiation is compiled for: X takes 16
// registers per unit, so wider K-slices get fewer warps.
__host__ __device__ constexpr int max_consumer_warps(int ku) { return ku <= 1 ? 20 : ku == 2 ? 12 : 8; }

// Partial dot products of one unit for NP row pairs (NP independent
// accumulator pairs, so the tensor-core chains overlap).  Both rows of a pair
// are always read: the stage buffer holds RS (even) rows, so the second row
// of a short last pair is stale data whose result is discarded.
// FULL: every lane's blocks lie inside K (K % 1024 == 0).  SB: scales are in
// the stage (bulk-copied) rather than read from global memory.
template <int NP, bool FULL, bool SB>
__device__ __forceinline__ void pairs_unit(float (&d)[NP][2][4], const uint8_t *st_codes,
                                           const uint8_t *st_scales, const uint8_t *g_scales,
                                           const int (&ra)[NP], int rows_i, int64_t KH,
                                           int64_t KB, int64_t kb, const uint32_t (&xr)[16]) {
  const bool lane_in = FULL || kb < KB;
#pragma unroll
  for (int p = 0; p < NP; ++p) {
    uint4 cw0 = make_uint4(0, 0, 0, 0), cw1 = make_uint4(0, 0, 0, 0);
    uint32_t sc0 = 0, sc1 = 0;
    if (lane_in) {
      const uint8_t *c = st_codes + ra[p] * KH + kb * 8;
      cw0 = *reinterpret_cast<const uint4 *>(c);
      cw1 = *reinterpret_cast<const uint4 *>(c + KH);
      if (SB) {
        const uint8_t *sp = st_scales + ra[p] * KB + kb;
        sc0 = *reinterpret_cast<const uint16_t *>(sp);
        sc1 = *reinterpret_cast<const uint16_t *>(sp + KB);
      } else {
        // global memory: never read past the stage's last row (the array may end there)
        const int rb = ra[p] + 1 < rows_i ? ra[p] + 1 : ra[p];
        sc0 = __ldg(reinterpret_cast<const uint16_t *>(g_scales + ra[p] * KB + kb));
        sc1 = __ldg(reinterpret_cast<const uint16_t *>(g_scales + rb * KB + kb));
      }
    }
    unit_mma(d[p][0], d[p][1], cw0, cw1, sc0, sc1, xr);
  }
}

template <int KU, bool FULL, bool SB>
__global__ void __launch_bounds__(kProducer + 32 * max_consumer_warps(KU), 1)
    gemv_m1_kernel(const M1Args a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int NS = a.nstages, RS = a.rows_per_stage, NWK = a.warps_per_row, RG = a.row_groups;
  const int RB = a.rows_per_block;
  const int n_cw = NWK * RG;  // consumer warps
  const int64_t KH = a.K / 2, KB = a.K / 16;
  const int n_units = (int)ceil_div(a.K, kUnitK);

  uint64_t *full = reinterpret_cast<uint64_t *>(smem);
  uint64_t *empty = full + kMaxStages;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + kMaxStages);
  float *red = reinterpret_cast<float *>(smem + kHeadBytes);  // [RB][NWK]
  float *wmax = red + (size_t)RB * NWK;                       // [32]
  const size_t red_bytes = ((size_t)RB * NWK + 32) * sizeof(float);
  uint8_t *stages = smem + kHeadBytes + ceil_div(red_bytes, 128) * 128;

  const int64_t G = gridDim.x;
  const int64_t row_begin = a.N * (int64_t)blockIdx.x / G;
  const int64_t row_end = a.N * ((int64_t)blockIdx.x + 1) / G;
  const int64_t n_st = ceil_div(row_end - row_begin, RS);

  // Programmatic dependent launch: the next kernel on the stream may start
  // as soon as SMs free up; its weight stream then overlaps this kernel's
  // tail.  Everything it reads before its own griddepcontrol.wait is weight
  // data, which no kernel in a decode step writes.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], n_cw);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (threadIdx.x < kProducer) {
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
      for (int64_t i = (issued > NS ? issued - NS : 0); i < issued; ++i)
        mbar_wait_bounded(&full[i % NS], (uint32_t)((i / NS) & 1), a.status);
    }
    return;
  }

  const int cw = (threadIdx.x - kProducer) >> 5;  // consumer warp
  const int ct = threadIdx.x - kProducer;
  const int lane = threadIdx.x & 31;
  const int rg = cw / NWK, wk = cw - rg * NWK;
  const int g = lane >> 2;
  const int u0 = wk * KU;  // first unit of this warp's K-slice

  // X (and Y) may belong to the previous kernel on the stream: wait for it
  // to complete (a no-op without programmatic dependent launch).  The
  // producer above does not wait -- it only reads the weight.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // ---- X for this warp's K-slice: lane's 32 elements per unit
  uint32_t xb[KU][16];
  uint32_t mx = 0;
#pragma unroll
  for (int j = 0; j < KU; ++j) {
    const int64_t k0 = (int64_t)(u0 + j) * kUnitK + 32 * lane;
#pragma unroll
    for (int i = 0; i < 16; ++i) xb[j][i] = 0u;
    if (u0 + j < n_units && k0 < a.K) {
      const uint4 *src = reinterpret_cast<const uint4 *>(a.x + k0);
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const uint4 q = __ldg(src + v);
        xb[j][4 * v] = q.x; xb[j][4 * v + 1] = q.y; xb[j][4 * v + 2] = q.z; xb[j][4 * v + 3] = q.w;
      }
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) mx = __vmaxu2(mx, xb[j][i] & 0x7FFF7FFFu);
  }
  mx = max(mx & 0xFFFFu, mx >> 16);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
  if (lane == 0) wmax[cw] = __uint_as_float(mx << 16);
  named_bar(1, n_cw * 32);
  float xmax = 0.0f;
  for (int w = 0; w < NWK; ++w) xmax = fmaxf(xmax, wmax[w]);
  int sh = 0;
  if (xmax > 0.0f && xmax < __int_as_float(0x7F800000)) {
    int e;
    frexpf(xmax, &e);
    sh = 15 - e;
  }
#pragma unroll
  for (int j = 0; j < KU; ++j)
#pragma unroll
    for (int i = 0; i < 16; ++i)
      xb[j][i] = f16x2_pack(ldexpf(bf16_bits_to_f32(xb[j][i] & 0xFFFFu), sh),
                            ldexpf(bf16_bits_to_f32(xb[j][i] >> 16), sh));
  const float out_scale = *a.tensor_scale;
  const float x_unscale = ldexpf(1.0f, -sh);
  const int dsel = g & 1;

  int64_t blk_row0 = row_begin;  // first row of the current row block
  for (int64_t i = 0; i < n_st; ++i) {
    const int s = (int)(i % NS);
    // warp-uniform: mma.sync and the shuffles below need all 32 lanes
    const bool ready =
        __all_sync(0xFFFFFFFFu, mbar_wait_bounded(&full[s], (uint32_t)((i / NS) & 1), a.status));
    if (!ready) *abort_flag = 1;
    const int64_t r0 = row_begin + i * RS;
    const int rows_i = (int)min((int64_t)RS, row_end - r0);
    const int rloc = (int)(r0 - blk_row0);  // stage offset within the row block
    const uint8_t *st_codes = stages + (size_t)s * a.stage_bytes;
    const uint8_t *st_scales = st_codes + a.codes_stage_bytes;
    const uint8_t *g_scales = a.scales + r0 * KB;
    const int n_pairs = ready ? (rows_i + 1) / 2 : 0;

    for (int p = rg; p < n_pairs; p += 2 * RG) {
      const bool two = p + RG < n_pairs;
      float v[4];
      if (two) {
        const int ra[2] = {2 * p, 2 * (p + RG)};
        float d[2][2][4] = {};
#pragma unroll
        for (int j = 0; j < KU; ++j) {
          const int u = u0 + j;
          if (u < n_units) {
            const int64_t kb = (int64_t)u * (kUnitK / 16) + 2 * lane;
            pairs_unit<2, FULL, SB>(d, st_codes, st_scales, g_scales, ra, rows_i, KH, KB, kb,
                                    xb[j]);
          }
        }
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          // register selects, not a runtime array index (which would put d on the stack)
          v[2 * q] = dsel ? d[q][0][1] + d[q][1][1] : d[q][0][0] + d[q][1][0];
          v[2 * q + 1] = dsel ? d[q][0][3] + d[q][1][3] : d[q][0][2] + d[q][1][2];
        }
      } else {
        const int ra[1] = {2 * p};
        float d[1][2][4] = {};
#pragma unroll
        for (int j = 0; j < KU; ++j) {
          const int u = u0 + j;
          if (u < n_units) {
            const int64_t kb = (int64_t)u * (kUnitK / 16) + 2 * lane;
            pairs_unit<1, FULL, SB>(d, st_codes, st_scales, g_scales, ra, rows_i, KH, KB, kb,
                                    xb[j]);
          }
        }
        v[0] = dsel ? d[0][0][1] + d[0][1][1] : d[0][0][0] + d[0][1][0];
        v[1] = dsel ? d[0][0][3] + d[0][1][3] : d[0][0][2] + d[0][1][2];
        v[2] = v[3] = 0.0f;
      }
      // D[g][g] (row 2p) and D[g+8][g] (row 2p+1) live in lane 4g + g/2, i.e.
      // lanes 9j (g = 2j) and 9j + 4 (g = 2j + 1).  XOR 4, then 9, then 18
      // gathers exactly those eight lanes into lane 0 (other lanes' sums are
      // never read).
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        v[q] += __shfl_xor_sync(0xFFFFFFFFu, v[q], 4);
        v[q] += __shfl_xor_sync(0xFFFFFFFFu, v[q], 9);
        v[q] += __shfl_xor_sync(0xFFFFFFFFu, v[q], 18);
      }
      if (lane == 0) {
        const int rr[4] = {2 * p, 2 * p + 1, 2 * (p + RG), 2 * (p + RG) + 1};
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (rr[q] < rows_i && (q < 2 || two)) red[(rloc + rr[q]) * NWK + wk] = v[q];
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);

    // End of a row block (or of the CTA's rows): fixed-order sums -> Y.
    const int64_t blk_end = min(blk_row0 + RB, row_end);
    if (r0 + rows_i >= blk_end || i + 1 == n_st) {
      named_bar(1, n_cw * 32);
      if (*abort_flag) return;
      const int nr = (int)(r0 + rows_i - blk_row0);
      for (int r = ct; r < nr; r += n_cw * 32) {
        float acc = 0.0f;
        for (int w = 0; w < NWK; ++w) acc += red[r * NWK + w];
        acc = (acc * x_unscale) * out_scale;
        a.y[blk_row0 + r] = __bfloat16_as_ushort(__float2bfloat16_rn(acc));
      }
      named_bar(1, n_cw * 32);
      blk_row0 = r0 + rows_i;
    }
  }
}

struct M1Plan {
  int KU, NWK, RG, RS, RB, NS, threads, scales_bulk;
  uint32_t stage_bytes, codes_stage_bytes;
  size_t smem;
};

bool make_m1_plan(int64_t N, int64_t K, M1Plan &p) {
  const int n_units = (int)ceil_div(K, kUnitK);
  // Fewest units per warp whose warps-per-row fit the instantiation (X
  // registers: 16 per unit).
  int KU = 1;
  while (KU <= 4 && ceil_div(n_units, KU) > max_consumer_warps(KU)) ++KU;
  if (KU > 4) return false;
  p.KU = KU;
  p.NWK = (int)ceil_div(n_units, KU);
  int RG = max_consumer_warps(KU) / p.NWK;
  if (RG < 1) RG = 1;
  p.RG = RG;
  p.threads = kProducer + 32 * p.NWK * p.RG;
  p.scales_bulk = (K % 256 == 0) ? 1 : 0;
  const int64_t row_bytes = K / 2 + (p.scales_bulk ? K / 16 : 0);
  // Each row group takes two row pairs per stage (two independent
  // accumulator sets per warp), more while a stage stays under ~40 KB.
  int64_t RS = 4 * p.RG;
  while (RS * 2 * row_bytes <= 40 * 1024 && RS < 128) RS *= 2;
  const int64_t rows_per_cta = ceil_div(N, num_sms());
  const int64_t cap = 2 * ceil_div(rows_per_cta, 2);
  if (RS > cap) RS = cap < 2 ? 2 : cap;
  p.RS = (int)RS;
  // Row block: the rows whose partial sums wait in shared memory (<= 24 KB).
  int64_t RB = (24 * 1024 / 4) / p.NWK;
  RB = (RB / RS) * RS;
  if (RB < RS) RB = RS;
  if (RB > ceil_div(rows_per_cta, RS) * RS) RB = ceil_div(rows_per_cta, RS) * RS;
  p.RB = (int)RB;
  p.codes_stage_bytes = (uint32_t)(ceil_div(RS * (K / 2), 128) * 128);
  const uint32_t sbytes = p.scales_bulk ? (uint32_t)(ceil_div(RS * (K / 16), 128) * 128) : 0u;
  p.stage_bytes = p.codes_stage_bytes + sbytes;
  auto total = [&](int ns) {
    const size_t red = ((size_t)p.RB * p.NWK + 32) * sizeof(float);
    return kHeadBytes + ceil_div(red, 128) * 128 + (size_t)ns * p.stage_bytes;
  };
  int NS = kMaxStages;
  while (NS > 2 && total(NS) > kSmemBudget) --NS;
  p.NS = NS;
  p.smem = total(NS);
  return p.smem <= 227 * 1024;
}

template <int KU, bool FULL, bool SB>
cudaError_t launch_m1(const M1Args &a, const M1Plan &p, int grid, cudaStream_t stream) {
  auto kern = gemv_m1_kernel<KU, FULL, SB>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(p.threads);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

bool gemv_m1_supported(int64_t N, int64_t K) {
  M1Plan p;
  return N >= 1 && K >= 64 && K % 64 == 0 && make_m1_plan(N, K, p);
}

cudaError_t launch_gemv_m1(const uint16_t *x, int64_t K, const uint8_t *codes,
                           const uint8_t *scales, const float *tensor_scale, int64_t N,
                           uint16_t *y, int32_t *status, cudaStream_t stream) {
  M1Plan p;
  if (!make_m1_plan(N, K, p)) return cudaErrorInvalidConfiguration;
  M1Args a;
  a.x = x;
  a.codes = codes;
  a.scales = scales;
  a.tensor_scale = tensor_scale;
  a.y = y;
  a.N = N;
  a.K = K;
  a.status = status;
  a.rows_per_stage = p.RS;
  a.nstages = p.NS;
  a.warps_per_row = p.NWK;
  a.row_groups = p.RG;
  a.rows_per_block = p.RB;
  a.scales_bulk = p.scales_bulk;
  a.stage_bytes = p.stage_bytes;
  a.codes_stage_bytes = p.codes_stage_bytes;
  int64_t grid = num_sms();
  if (grid > N) grid = N;
  const bool full = (K % kUnitK) == 0;
#define IMPFP4_KU(ku)                                                               \
  case ku:                                                                          \
    if (full && p.scales_bulk) return launch_m1<ku, true, true>(a, p, (int)grid, stream); \
    if (p.scales_bulk) return launch_m1<ku, false, true>(a, p, (int)grid, stream);  \
    return launch_m1<ku, false, false>(a, p, (int)grid, stream);
  switch (p.KU) {
    IMPFP4_KU(1)
    IMPFP4_KU(2)
    IMPFP4_KU(3)
    IMPFP4_KU(4)
  }
#undef IMPFP4_KU
  return cudaErrorInvalidConfiguration;
}

}  // namespace impfp4
