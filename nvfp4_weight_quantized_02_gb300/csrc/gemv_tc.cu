// Decode GEMV on the tensor cores, one pass per tile of MT in {1, 2, 4, 8}
// rows of X: y[m][n] = s * sum_k x[m][k] * e2m1(c[n][k]) * e4m3(sb[n][k/16]).
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
//    f16 x f16 -> f32) with a block-group diagonal.  With G = 8 / MT groups,
//    one "unit" covers 128 G values of k and a row set of R = 2 MT weight
//    rows.  Lane L = 4g + t takes group a = g % G and owns the two 16-element
//    blocks 2(4a + t), 2(4a + t) + 1 of the unit:
//      A row g     = weight row g / G      of the row set, at group a's k,
//      A row g + 8 = weight row g / G + MT of the row set, at group a's k,
//      B column g  = X row g / G, at group a's k,
//    so D[i][j] is a partial dot product exactly when i % G == j % G, and
//    summing those over the G groups (log2 G shuffle steps: XOR 4, 9, 18)
//    gives weight row x X row.  Each lane reads 16 contiguous code bytes per
//    weight row (the lanes of one row read 64 G contiguous bytes: no bank
//    conflicts).  Eight mma steps cover the unit (step s takes elements
//    4(s%4)..4(s%4)+3 of block 2(4a + t) + s/4 in every lane).  At MT = 1
//    two of the 32 entries of D are used, at MT = 8 all of them: the decode
//    work per weight is the same, shared by MT rows of X.
//  * A fragments: cvt.rn.f16x2.e2m1x2 per code byte, multiplied (HMUL2) by
//    the block's E4M3 scale (cvt.rn.f16x2.e4m3x2).  e2m1 * e4m3 has at most
//    6 significant bits and lies in [2^-10, 2688], so it is exact in f16.
//  * B fragments: each warp owns a fixed K-slice and keeps X for it in
//    registers as f16 (16 registers per unit), each X row scaled by one power
//    of two 2^sh per call so that its max|x| lies in [2^14, 2^15): exact for
//    every element within 2^24 of the row's largest (smaller ones round to
//    f16 subnormals: an absolute error below max|x| * 2^-39 per element).
//    The factor is undone in fp32 at the end.
//  * Products are exact; sums are fp32 (tensor-core accumulation across the
//    warp's units, then the shuffle butterfly, then a fixed-order sum of the
//    per-warp partials), times the tensor scale, rounded to bf16.  No step
//    depends on timing, so results are bitwise reproducible.
//  * Rows of X beyond 8 take further passes; MT shrinks where X for the
//    tile does not fit the consumer warps' registers (large K).
#include "gemv.cuh"

namespace impfp4 {

namespace {

constexpr int kProducer = 32;
constexpr int kMaxStages = 8;
constexpr size_t kSmemBudget = 200 * 1024;
constexpr size_t kHeadBytes = 2 * kMaxStages * sizeof(uint64_t) + 16;

struct M1Args {
  const uint16_t *x;
  int64_t ldx;
  int M;  // rows of X in this pass (<= MT); the others are zero
  int64_t ldy;
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

// One unit: A rows g and g + 8.  cw0/cw1: the lane's 16 code bytes of
// each; sc0/sc1: its two scale bytes of each; xr: the lane's 32 X
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
// registers per unit, so wider K-slices get fewer warps (the launch bound
// leaves each thread >= 120 registers from KU = 2 on).
__host__ __device__ constexpr int max_consumer_warps(int ku) {
  return ku <= 1 ? 20 : ku == 2 ? 16 : ku == 3 ? 12 : 10;
}

// Block groups per MMA: with MT rows of X, A rows are (weight row, group) for
// 2*MT weight rows x G groups and B columns (X row, group) for MT rows x G.
template <int MT> struct TileCfg {
  static constexpr int G = 8 / MT;          // block groups per MMA
  static constexpr int UNIT_K = 128 * G;    // K elements per unit
  static constexpr int R = 2 * MT;          // weight rows per row set
};

// Partial products of one unit for NP row sets (NP independent accumulator
// pairs, so the tensor-core chains overlap).  Lane (g, t) reads 16 code bytes
// of weight rows lo and lo + MT of each row set; both rows are always read
// (the stage buffer holds RS rows, a multiple of the row-set size), and
// results of rows past the stage are discarded.
template <int NP, int MT, bool FULL, bool SB>
__device__ __forceinline__ void sets_unit(float (&d)[NP][2][4], const uint8_t *st_codes,
                                          const uint8_t *st_scales, const uint8_t *g_scales,
                                          const int (&rlo)[NP], int rows_i, int64_t KH,
                                          int64_t KB, int64_t kb, const uint32_t (&xr)[16]) {
  const bool lane_in = FULL || kb < KB;
#pragma unroll
  for (int p = 0; p < NP; ++p) {
    uint4 cw0 = make_uint4(0, 0, 0, 0), cw1 = make_uint4(0, 0, 0, 0);
    uint32_t sc0 = 0, sc1 = 0;
    if (lane_in) {
      const uint8_t *c = st_codes + rlo[p] * KH + kb * 8;
      cw0 = *reinterpret_cast<const uint4 *>(c);
      cw1 = *reinterpret_cast<const uint4 *>(c + MT * KH);
      if (SB) {
        const uint8_t *sp = st_scales + rlo[p] * KB + kb;
        sc0 = *reinterpret_cast<const uint16_t *>(sp);
        sc1 = *reinterpret_cast<const uint16_t *>(sp + MT * KB);
      } else {
        // global memory: never read past the stage's last row (the array may end there)
        const int r0 = rlo[p] < rows_i ? rlo[p] : rows_i - 1;
        const int r1 = rlo[p] + MT < rows_i ? rlo[p] + MT : rows_i - 1;
        sc0 = __ldg(reinterpret_cast<const uint16_t *>(g_scales + r0 * KB + kb));
        sc1 = __ldg(reinterpret_cast<const uint16_t *>(g_scales + r1 * KB + kb));
      }
    }
    unit_mma(d[p][0], d[p][1], cw0, cw1, sc0, sc1, xr);
  }
}

template <int MT, int KU, bool FULL, bool SB>
__global__ void __launch_bounds__(kProducer + 32 * max_consumer_warps(KU), 1)
    gemv_tc_kernel(const M1Args a) {
  using C = TileCfg<MT>;
  constexpr int G = C::G, UNIT_K = C::UNIT_K, R = C::R;
  extern __shared__ __align__(128) uint8_t smem[];
  const int NS = a.nstages, RS = a.rows_per_stage, NWK = a.warps_per_row, RG = a.row_groups;
  const int RB = a.rows_per_block;
  const int n_cw = NWK * RG;  // consumer warps
  const int64_t KH = a.K / 2, KB = a.K / 16;
  const int n_units = (int)ceil_div(a.K, UNIT_K);

  uint64_t *full = reinterpret_cast<uint64_t *>(smem);
  uint64_t *empty = full + kMaxStages;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + kMaxStages);
  float *red = reinterpret_cast<float *>(smem + kHeadBytes);  // [RB][MT][NWK]
  float *wmax = red + (size_t)RB * MT * NWK;                  // [32][MT]
  float *unscale = wmax + 32 * MT;                            // [MT]
  const size_t red_bytes = ((size_t)RB * MT * NWK + 33 * MT) * sizeof(float);
  uint8_t *stages = smem + kHeadBytes + ceil_div(red_bytes, 128) * 128;

  const int64_t GR = gridDim.x;
  const int64_t row_begin = a.N * (int64_t)blockIdx.x / GR;
  const int64_t row_end = a.N * ((int64_t)blockIdx.x + 1) / GR;
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
  const int g = lane >> 2, t = lane & 3;
  const int grp = g % G;      // block group of this lane
  const int m_lane = g / G;   // X row of this lane's B column = weight row offset of A row g
  const int lane_blk = 2 * (4 * grp + t);  // first of the lane's two blocks in a unit
  const int u0 = wk * KU;     // first unit of this warp's K-slice

  // X (and Y) may belong to the previous kernel on the stream: wait for it
  // to complete (a no-op without programmatic dependent launch).  The
  // producer above does not wait -- it only reads the weight.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // ---- X for this warp's K-slice: row m_lane, the lane's 32 elements per unit
  uint32_t xb[KU][16];
  uint32_t mx = 0;
#pragma unroll
  for (int j = 0; j < KU; ++j) {
    const int64_t k0 = (int64_t)(u0 + j) * UNIT_K + 16 * lane_blk;
#pragma unroll
    for (int i = 0; i < 16; ++i) xb[j][i] = 0u;
    if (u0 + j < n_units && k0 < a.K && m_lane < a.M) {
      const uint4 *src = reinterpret_cast<const uint4 *>(a.x + (int64_t)m_lane * a.ldx + k0);
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
  // max over the lanes holding the same X row (lanes 4G*m .. 4G*m + 4G-1)
#pragma unroll
  for (int o = 1; o < 4 * G; o <<= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
  if ((lane & (4 * G - 1)) == 0) wmax[cw * MT + m_lane] = __uint_as_float(mx << 16);
  named_bar(1, n_cw * 32);
  float xmax = 0.0f;
  for (int w = 0; w < NWK; ++w) xmax = fmaxf(xmax, wmax[w * MT + m_lane]);
  int sh = 0;
  if (xmax > 0.0f && xmax < __int_as_float(0x7F800000)) {
    int e;
    frexpf(xmax, &e);
    sh = 15 - e;
  }
  if (cw == 0 && (lane & (4 * G - 1)) == 0) unscale[m_lane] = ldexpf(1.0f, -sh);
#pragma unroll
  for (int j = 0; j < KU; ++j)
#pragma unroll
    for (int i = 0; i < 16; ++i)
      xb[j][i] = f16x2_pack(ldexpf(bf16_bits_to_f32(xb[j][i] & 0xFFFFu), sh),
                            ldexpf(bf16_bits_to_f32(xb[j][i] >> 16), sh));
  const float out_scale = *a.tensor_scale;

  // Which accumulator register holds a useful sum in this lane: column
  // j = 2t + u pairs with A row g when j and g fall in the same block group.
  const int u_sel = (grp - 2 * t) & (G - 1);
  const bool useful = G == 1 || u_sel < 2;
  const int m_out = G == 1 ? 0 : (2 * t + u_sel) / G;  // X row of the useful column
  const bool writer = G == 1 || (grp == 0 && useful);

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
    const int n_sets = ready ? (rows_i + R - 1) / R : 0;

    for (int p = rg; p < n_sets; p += 2 * RG) {
      const bool two = p + RG < n_sets;
      float dd[2][2][4] = {};
      const int rlo[2] = {p * R + m_lane, (p + RG) * R + m_lane};
#pragma unroll
      for (int j = 0; j < KU; ++j) {
        const int u = u0 + j;
        if (u < n_units) {  // warp-uniform; lanes past K feed zeros to the mma
          const int64_t kb = (int64_t)u * (UNIT_K / 16) + lane_blk;
          if (two)
            sets_unit<2, MT, FULL, SB>(dd, st_codes, st_scales, g_scales, rlo, rows_i, KH, KB,
                                       kb, xb[j]);
          else
            sets_unit<1, MT, FULL, SB>(*reinterpret_cast<float(*)[1][2][4]>(&dd[0]), st_codes,
                                       st_scales, g_scales,
                                       *reinterpret_cast<const int(*)[1]>(&rlo[0]), rows_i, KH,
                                       KB, kb, xb[j]);
        }
      }
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        if (q == 1 && !two) break;  // warp-uniform
        const float (&d0)[4] = dd[q][0];
        const float (&d1)[4] = dd[q][1];
        if (G == 1) {
          // every entry useful: weight rows g and g+8, X rows 2t and 2t+1
          const int rb = (p + q * RG) * R;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int row = rb + g + (k >= 2 ? 8 : 0);
            const int m = 2 * t + (k & 1);
            if (row < rows_i) red[((size_t)(rloc + row) * MT + m) * NWK + wk] = d0[k] + d1[k];
          }
        } else {
          // register selects, not a runtime array index (which would put d on the stack)
          float vlo = u_sel ? d0[1] + d1[1] : d0[0] + d1[0];
          float vhi = u_sel ? d0[3] + d1[3] : d0[2] + d1[2];
          vlo = useful ? vlo : 0.0f;
          vhi = useful ? vhi : 0.0f;
          // the G lanes of one output: XOR 4 (G >= 2), then 9 (G >= 4), then 18 (G == 8)
          vlo += __shfl_xor_sync(0xFFFFFFFFu, vlo, 4);
          vhi += __shfl_xor_sync(0xFFFFFFFFu, vhi, 4);
          if (G >= 4) {
            vlo += __shfl_xor_sync(0xFFFFFFFFu, vlo, 9);
            vhi += __shfl_xor_sync(0xFFFFFFFFu, vhi, 9);
          }
          if (G == 8) {
            vlo += __shfl_xor_sync(0xFFFFFFFFu, vlo, 18);
            vhi += __shfl_xor_sync(0xFFFFFFFFu, vhi, 18);
          }
          if (writer) {
            const int rb = (p + q * RG) * R + m_lane;
            if (rb < rows_i) red[((size_t)(rloc + rb) * MT + m_out) * NWK + wk] = vlo;
            if (rb + MT < rows_i) red[((size_t)(rloc + rb + MT) * MT + m_out) * NWK + wk] = vhi;
          }
        }
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
      for (int o = ct; o < nr * MT; o += n_cw * 32) {
        const int r = o / MT, m = o - r * MT;
        if (m < a.M) {
          float acc = 0.0f;
          for (int w = 0; w < NWK; ++w) acc += red[((size_t)r * MT + m) * NWK + w];
          acc = (acc * unscale[m]) * out_scale;
          a.y[(int64_t)m * a.ldy + blk_row0 + r] = __bfloat16_as_ushort(__float2bfloat16_rn(acc));
        }
      }
      named_bar(1, n_cw * 32);
      blk_row0 = r0 + rows_i;
    }
  }
}

struct M1Plan {
  int MT, KU, NWK, RG, RS, RB, NS, threads, scales_bulk;
  uint32_t stage_bytes, codes_stage_bytes;
  size_t smem;
};

bool make_tc_plan(int MT, int64_t N, int64_t K, M1Plan &p) {
  const int unit_k = 128 * (8 / MT);
  const int n_units = (int)ceil_div(K, unit_k);
  // Fewest units per warp whose warps-per-row fit the instantiation (X
  // registers: 16 per unit).
  int KU = 1;
  while (KU <= 4 && ceil_div(n_units, KU) > max_consumer_warps(KU)) ++KU;
  if (KU > 4) return false;
  p.MT = MT;
  p.KU = KU;
  p.NWK = (int)ceil_div(n_units, KU);
  int RG = max_consumer_warps(KU) / p.NWK;
  if (RG < 1) RG = 1;
  p.RG = RG;
  p.threads = kProducer + 32 * p.NWK * p.RG;
  p.scales_bulk = (K % 256 == 0) ? 1 : 0;
  const int64_t row_bytes = K / 2 + (p.scales_bulk ? K / 16 : 0);
  const int R = 2 * MT;
  // Each row group takes two row sets per stage (two independent
  // accumulator sets per warp), more while a stage stays under ~40 KB.
  int64_t RS = 2 * R * p.RG;
  while (RS * 2 * row_bytes <= 40 * 1024 && RS < 128) RS *= 2;
  const int64_t rows_per_cta = ceil_div(N, num_sms());
  const int64_t cap = R * ceil_div(rows_per_cta, R);
  if (RS > cap) RS = cap;
  if (RS * row_bytes > 96 * 1024) return false;
  p.RS = (int)RS;
  // Row block: the rows whose partial sums wait in shared memory (<= 24 KB).
  int64_t RB = (24 * 1024 / 4) / (p.NWK * MT);
  RB = (RB / RS) * RS;
  if (RB < RS) RB = RS;
  if (RB > ceil_div(rows_per_cta, RS) * RS) RB = ceil_div(rows_per_cta, RS) * RS;
  p.RB = (int)RB;
  p.codes_stage_bytes = (uint32_t)(ceil_div(RS * (K / 2), 128) * 128);
  const uint32_t sbytes = p.scales_bulk ? (uint32_t)(ceil_div(RS * (K / 16), 128) * 128) : 0u;
  p.stage_bytes = p.codes_stage_bytes + sbytes;
  auto total = [&](int ns) {
    const size_t red = ((size_t)p.RB * MT * p.NWK + 33 * MT) * sizeof(float);
    return kHeadBytes + ceil_div(red, 128) * 128 + (size_t)ns * p.stage_bytes;
  };
  int NS = kMaxStages;
  while (NS > 2 && total(NS) > kSmemBudget) --NS;
  p.NS = NS;
  p.smem = total(NS);
  return p.smem <= 227 * 1024;
}

template <int MT, int KU, bool FULL, bool SB>
cudaError_t launch_tc(const M1Args &a, const M1Plan &p, int grid, cudaStream_t stream) {
  auto kern = gemv_tc_kernel<MT, KU, FULL, SB>;
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

template <int MT>
cudaError_t dispatch_tc(const M1Args &a, const M1Plan &p, int grid, cudaStream_t stream) {
  const bool full = (a.K % (128 * (8 / MT))) == 0;
#define IMPFP4_KU(ku)                                                                    \
  case ku:                                                                               \
    if (full && p.scales_bulk) return launch_tc<MT, ku, true, true>(a, p, grid, stream); \
    if (p.scales_bulk) return launch_tc<MT, ku, false, true>(a, p, grid, stream);        \
    return launch_tc<MT, ku, false, false>(a, p, grid, stream);
  switch (p.KU) {
    IMPFP4_KU(1)
    IMPFP4_KU(2)
    IMPFP4_KU(3)
    IMPFP4_KU(4)
  }
#undef IMPFP4_KU
  return cudaErrorInvalidConfiguration;
}

// Rows of X per pass: the largest tile in {8, 4, 2, 1} that has a plan, not
// above the rows left rounded up to a power of two.
int tc_pass_tile(int64_t M_left, int64_t N, int64_t K, M1Plan &p) {
  const int want = M_left >= 5 ? 8 : M_left >= 3 ? 4 : (int)M_left;
  for (int mt = want; mt >= 1; mt /= 2)
    if (make_tc_plan(mt, N, K, p)) return mt;
  return 0;
}

}  // namespace

int gemv_tc_launches(int64_t M, int64_t N, int64_t K) {
  if (M < 1 || M > kDecodeMaxM || N < 1 || K < 64 || K % 64) return 0;
  int passes = 0;
  for (int64_t m0 = 0; m0 < M; ++passes) {
    M1Plan p;
    const int mt = tc_pass_tile(M - m0, N, K, p);
    if (mt == 0) return 0;
    m0 += mt;
  }
  return passes;
}

bool gemv_tc_supported(int64_t M, int64_t N, int64_t K) { return gemv_tc_launches(M, N, K) > 0; }

cudaError_t launch_gemv_tc(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                           const uint8_t *codes, const uint8_t *scales, const float *tensor_scale,
                           int64_t N, uint16_t *y, int64_t ldy, int32_t *status,
                           cudaStream_t stream) {
  int64_t grid = num_sms();
  if (grid > N) grid = N;
  for (int64_t m0 = 0; m0 < M;) {
    M1Plan p;
    const int mt = tc_pass_tile(M - m0, N, K, p);
    if (mt == 0) return cudaErrorInvalidConfiguration;
    M1Args a;
    a.x = x + m0 * ldx;
    a.ldx = ldx;
    a.M = (int)((M - m0) < mt ? (M - m0) : mt);
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
    a.warps_per_row = p.NWK;
    a.row_groups = p.RG;
    a.rows_per_block = p.RB;
    a.scales_bulk = p.scales_bulk;
    a.stage_bytes = p.stage_bytes;
    a.codes_stage_bytes = p.codes_stage_bytes;
    cudaError_t e = cudaErrorInvalidConfiguration;
    switch (mt) {
      case 1: e = dispatch_tc<1>(a, p, (int)grid, stream); break;
      case 2: e = dispatch_tc<2>(a, p, (int)grid, stream); break;
      case 4: e = dispatch_tc<4>(a, p, (int)grid, stream); break;
      case 8: e = dispatch_tc<8>(a, p, (int)grid, stream); break;
    }
    if (e != cudaSuccess) return e;
    m0 += mt;
  }
  return cudaSuccess;
}

}  // namespace impfp4
