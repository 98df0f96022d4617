// Prefill NVFP4 GEMM on the block-scaled FP4 tensor cores of sm_103a:
//   Y[M][N] = s_x * s_w * sum_k (e2m1_x * e4m3_x)[m][k] * (e2m1_w * e4m3_w)[n][k]
// with X already quantized to NVFP4 by the same recipe as W.  Prefill is the
// compute-bound phase (imp README, "How it works"; "1. The big picture",
// section "Two phases with very different costs"), so it runs on
// tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X: FP4 x FP4 products
// with one E4M3 scale per 16 elements of each operand, fp32 accumulation in
// tensor memory.
//
// Structure (one CTA per SM, persistent over 128 x 256 output tiles):
//  * warp 0, one thread: TMA producer.  Per K-stage of 256 elements it loads
//    the X tile (128 rows x 128 bytes) with a 2-D tensor copy in the 128-byte
//    swizzle, the W tile (256 rows x 128 bytes) the same way -- or, for a
//    weight in the tile layout (quantize.cuh), as two contiguous 16 KB bulk
//    copies of the same swizzled image -- and the matching block scales
//    (already in the 512-byte atom layout) with bulk copies, into a 4-deep
//    shared-memory ring.
//  * warp 10, one thread: per stage, twelve tcgen05.cp (per 64-element K
//    step: the scales of the X rows and of the two 128-row halves of the W
//    tile) into the stage's own bank of tensor-memory columns, then a
//    tcgen05.commit that tells the MMA warp the bank is ready.  A copy costs
//    the issuing thread about as much as an MMA, so issuing both from one
//    thread left the tensor pipe idle half of the time.
//  * warp 1: allocates 512 tensor-memory columns; one thread issues, per
//    stage, four tcgen05.mma (M = 128, N = 256, K = 64) accumulating into
//    columns 0..255; tcgen05.commit releases each ring stage and, at the end
//    of a tile, signals the epilogue.
//  * warps 2..9: epilogue.  Each thread owns half of one accumulator row
//    (its warp's 32-lane quarter of tensor memory, 128 of the 256 columns),
//    reads it with tcgen05.ld, multiplies by s_x * s_w, rounds to bf16, hands
//    the accumulator back, then stores to Y while the next tile's MMAs run.
// Every wait is bounded; on a timeout the kernel reports IMP_DEV_TIMEOUT,
// drains its own copies and MMAs, frees tensor memory and returns.
#include <cstring>

#include "gemm_tcgen05.cuh"
#include "quantize.cuh"
#include "tma.cuh"

namespace impfp4 {

namespace {

constexpr int BM = 128, BN = 256, BK = 256;  // BK in elements (128 bytes of codes)
constexpr int MMA_K = 64;
constexpr int KSTEPS = BK / MMA_K;  // 4 MMAs per stage
constexpr int NSTAGE = 4;
constexpr uint32_t A_BYTES = BM * BK / 2;                    // 16 KB
constexpr uint32_t B_BYTES = BN * BK / 2;                    // 32 KB
constexpr uint32_t SFA_BYTES = (BM / 128) * KSTEPS * 512;    // 2 KB
constexpr uint32_t SFB_BYTES = (BN / 128) * KSTEPS * 512;    // 4 KB
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
constexpr uint32_t OFF_B = A_BYTES, OFF_SFA = A_BYTES + B_BYTES, OFF_SFB = OFF_SFA + SFA_BYTES;
// warp 0 TMA, warp 1 MMA, warps 2..9 epilogue, warps 10..12 scale copies
constexpr int kScaleWarp0 = 10, kScaleWarps = 4;  // one per tensor-memory lane quarter
constexpr int kThreads = 32 * (kScaleWarp0 + kScaleWarps);
constexpr int kEpiThreads = 256;
constexpr int kEpiCols = 128;  // accumulator columns per epilogue warp
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TMEM_D = 0;     // accumulator: columns 0..255
constexpr uint32_t TMEM_SF = 256;  // scales: 12 columns per K step (X 4, W 8), a bank of 48 per ring stage
static_assert(TMEM_SF + 48 * NSTAGE <= TMEM_COLS, "tensor memory plan");
constexpr size_t kBarBytes = 256;
constexpr size_t kSmemBytes = 1024 + NSTAGE * (size_t)STAGE_BYTES + kBarBytes;

struct GemmArgs {
  const uint8_t *sfa;  // X block scales, atom layout
  const uint8_t *sfb;  // W block scales, atom layout
  const uint8_t *w_tiles;  // W codes in the 16 KB tile layout, or nullptr: TMA on row-major codes
  const float *s_x, *s_w;
  uint16_t *y;
  int64_t ldy;
  int M, N, K;
  int32_t *status;
  // stream-K (with a workspace): per-tile counters and per-CTA partial tiles
  unsigned __int128 *cnt;  // [tiles]
  float *part;             // [CTA][first/last segment][128 rows][256 columns]
  unsigned long long epoch;
  int stream_k;
  // SwiGLU (w2_tiles set; whole tiles, tiled weights): a tile's 256 W rows
  // are 128 rows of the gate weight (w_tiles, sfb, s_w) and the same 128
  // rows of the up weight (w2_tiles, sfb2, s_w2); the epilogue writes
  // h = silu(g) * u for 128 columns and folds max|h| (bf16 magnitude bits)
  // into *h_amax.
  const uint8_t *w2_tiles, *sfb2;
  const float *s_w2;
  uint32_t *h_amax;
};

// The work of one CTA as segments (tile, K-stage range), in processing order.
//  * Without a workspace: whole tiles blockIdx.x, + gridDim.x, ...
//  * Stream-K: the (tile, K stage) sequence, tile-major, cut into gridDim.x
//    equal contiguous ranges; a CTA's range covers whole tiles and at most two
//    partial ones, which it processes first (its first segment, then its
//    last) so that the split tiles' fix-ups overlap its whole tiles.
struct Sched {
  int sk, n_tiles, n_ks, G, c;
  int64_t total, g0, g1;
  int n_seg;
  __device__ Sched(int sk_, int n_tiles_, int n_ks_)
      : sk(sk_), n_tiles(n_tiles_), n_ks(n_ks_), G((int)gridDim.x), c((int)blockIdx.x) {
    total = (int64_t)n_tiles * n_ks;
    if (sk) {
      g0 = total * c / G;
      g1 = total * (c + 1) / G;
      n_seg = g1 > g0 ? (int)((g1 - 1) / n_ks - g0 / n_ks) + 1 : 0;
    } else {
      g0 = g1 = 0;
      n_seg = c < n_tiles ? (n_tiles - 1 - c) / G + 1 : 0;
    }
  }
  // natural (K-ordered) index of the segment processed at position jj
  __device__ int natural(int jj) const {
    if (!sk || n_seg < 2) return jj;
    return jj == 0 ? 0 : jj == 1 ? n_seg - 1 : jj - 1;
  }
  __device__ void seg(int jj, int &tile, int &k0, int &k1) const {
    const int j = natural(jj);
    if (!sk) {
      tile = c + j * G;
      k0 = 0;
      k1 = n_ks;
      return;
    }
    tile = (int)(g0 / n_ks) + j;
    const int64_t b = (int64_t)tile * n_ks;
    k0 = (int)((g0 > b ? g0 : b) - b);
    k1 = (int)((g1 < b + n_ks ? g1 : b + n_ks) - b);
  }
  // CTA owning unit g (stream-K)
  __device__ int owner(int64_t g) const { return (int)(((g + 1) * G - 1) / total); }
  // partial slot CTA cc uses for tile t: its first segment 0, its last 1
  __device__ int slot_of(int cc, int t) const {
    const int64_t b0 = total * cc / G;
    return (b0 / n_ks == t) ? 0 : 1;
  }
};

// ---- tcgen05 helpers (inline PTX) --------------------------------------------

// Shared-memory matrix descriptor (tcgen05): start address, leading and
// stride byte offsets (16-byte units), descriptor version 1, layout type.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                              uint32_t layout) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // version
  d |= (uint64_t)(layout & 7u) << 61;
  return d;
}
constexpr uint32_t kLayoutNone = 0, kLayoutSw128 = 2;

// Instruction descriptor, kind::mxf4nvf4 with E4M3 block scales: A and B are
// E2M1 (format 1), both K-major, N >> 3 at bit 17, M >> 4 at bit 24.
constexpr uint32_t kIdesc = (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                            ((uint32_t)(BM >> 4) << 24);

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_cp_sf(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, "
      "[%5], [%6], p;\n}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tc_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Four consecutive tensor-memory columns of this warp's 32 lanes (one 32-bit
// value per lane and column).
__device__ __forceinline__ void tc_st4(uint32_t taddr, uint4 v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr), "r"(v.x),
               "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&h);
}

// 32 bf16 (16 packed pairs, low half first) to Y[m][n .. n + 31] (columns
// >= N and rows >= M are not written).
__device__ __forceinline__ void store_packed_bf16(const GemmArgs &a, int64_t m, int n,
                                                  const uint32_t (&p)[16]) {
  if (m >= a.M) return;
  uint16_t *dst = a.y + m * a.ldy + n;
  if (n + 32 <= a.N) {
    uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
    for (int i = 0; i < 4; ++i) d4[i] = make_uint4(p[4 * i], p[4 * i + 1], p[4 * i + 2], p[4 * i + 3]);
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (n + 2 * i < a.N) dst[2 * i] = (uint16_t)(p[i] & 0xFFFFu);
      if (n + 2 * i + 1 < a.N) dst[2 * i + 1] = (uint16_t)(p[i] >> 16);
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_mxf4_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB, const GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + NSTAGE * STAGE_BYTES);
  uint64_t *empty = full + NSTAGE;
  uint64_t *accf = empty + NSTAGE;  // accumulator ready for the epilogue
  uint64_t *acce = accf + 1;        // accumulator drained by the epilogue
  uint64_t *sff = acce + 1;         // [NSTAGE] a stage's scales copied to tensor memory
  uint64_t *part_done = sff + NSTAGE;  // epilogue warps stored a split tile's partials
  uint64_t *flag_ready = part_done + 1;  // the tile's count is known
  uint64_t *drain = flag_ready + 1;      // the MMA thread's last MMAs completed
  volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(drain + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  volatile int *last_flag = abort_flag + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool swiglu = a.w2_tiles != nullptr;
  const int bn_out = swiglu ? BN / 2 : BN;  // output columns per tile
  const int MB = (a.M + BM - 1) / BM, NB = (a.N + bn_out - 1) / bn_out;
  const int n_tiles = MB * NB;
  const int n_ks = (a.K + BK - 1) / BK;
  const int KA = a.K / 64;  // scale atoms per 128-row block
  const Sched sch(a.stream_k, n_tiles, n_ks);

  if (threadIdx.x == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&sff[s], kScaleWarps);
    }
    mbar_init(accf, 1);
    mbar_init(acce, kEpiThreads);
    mbar_init(part_done, kEpiThreads / 32);
    mbar_init(flag_ready, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    if (!a.w_tiles) prefetch_tmap(&tmB);
  }
  // Launched with programmatic dependent launch: the launch and the set-up
  // above overlap the previous kernel (X's quantizer).  Nothing is read, Y
  // is not written and tensor memory is not claimed (the previous kernel
  // may still need to allocate it) before that kernel has finished.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(const_cast<uint32_t *>(tmem_slot))),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------ TMA producer
    if (lane == 0) {
      int64_t it = 0;
      bool ok = true;
      for (int jj = 0; ok && jj < sch.n_seg; ++jj) {
        int t, k0, k1;
        sch.seg(jj, t, k0, k1);
        const int mb = t % MB, nb = t / MB;
        for (int ks = k0; ks < k1; ++ks, ++it) {
          const int s = (int)(it % NSTAGE);
          if (it >= NSTAGE &&
              !mbar_wait_bounded(&empty[s], (uint32_t)(((it / NSTAGE) - 1) & 1), a.status)) {
            ok = false;
            break;
          }
          const int natoms = min(KSTEPS, KA - ks * KSTEPS);
          uint8_t *st = smem + (size_t)s * STAGE_BYTES;
          mbar_arrive_expect_tx(&full[s], A_BYTES + B_BYTES + 3u * natoms * 512u);
          tma_load_2d(st, &tmA, ks * (BK / 2), mb * BM, &full[s]);
          // the two 128-row halves of the W tile: 128-row blocks 2 nb and
          // 2 nb + 1 of W, or (SwiGLU) block nb of the gate and of the up weight
          const int64_t blk0 = swiglu ? nb : 2 * nb, blk1 = swiglu ? nb : 2 * nb + 1;
          const uint8_t *w1 = swiglu ? a.w2_tiles : a.w_tiles;
          const uint8_t *sf1 = swiglu ? a.sfb2 : a.sfb;
          if (a.w_tiles) {
            // two 128-row tiles, each stored as its swizzled shared-memory image
            const int64_t nch = (a.K + BK - 1) / BK;
            bulk_g2s(st + OFF_B, a.w_tiles + (blk0 * nch + ks) * 16384, 16384u, &full[s]);
            bulk_g2s(st + OFF_B + 16384, w1 + (blk1 * nch + ks) * 16384, 16384u, &full[s]);
          } else {
            tma_load_2d(st + OFF_B, &tmB, ks * (BK / 2), nb * BN, &full[s]);
          }
          const int64_t atom0 = (int64_t)ks * KSTEPS;
          bulk_g2s(st + OFF_SFA, a.sfa + ((int64_t)mb * KA + atom0) * 512, natoms * 512u,
                   &full[s]);
          bulk_g2s(st + OFF_SFB, a.sfb + (blk0 * KA + atom0) * 512, natoms * 512u, &full[s]);
          bulk_g2s(st + OFF_SFB + 2048, sf1 + (blk1 * KA + atom0) * 512, natoms * 512u,
                   &full[s]);
        }
      }
      if (!ok) {
        *abort_flag = 1;
        // drain: the last NSTAGE issued stages must land before shared memory is released
        for (int64_t i = (it > NSTAGE ? it - NSTAGE : 0); i < it; ++i)
          mbar_wait_bounded(&full[i % NSTAGE], (uint32_t)((i / NSTAGE) & 1), a.status);
      }
    }
  } else if (warp == 1) {
    // ------------------------------ MMA issuer
    // One thread, so every scalar instruction of this loop sits between two
    // MMAs: stage index and phase rotate instead of being divided out, and
    // each stage's descriptors are the stage-0 ones plus one offset (the
    // 14-bit start-address field cannot carry: shared addresses < 256 KB).
    if (lane == 0) {
      const uint64_t dA0 = smem_desc(smem_u32(smem), 16, 1024, kLayoutSw128);
      const uint64_t dB0 = smem_desc(smem_u32(smem + OFF_B), 16, 1024, kLayoutSw128);
      uint32_t s = 0, phase = 0;  // ring position of the next stage
      int tile_iter = 0;
      bool ok = true;
      for (int jj = 0; ok && jj < sch.n_seg; ++jj, ++tile_iter) {
        int t, k0, k1;
        sch.seg(jj, t, k0, k1);
        if (tile_iter > 0 &&
            !mbar_wait_bounded(acce, (uint32_t)((tile_iter - 1) & 1), a.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int ks = k0; ks < k1; ++ks) {
          // No shared-memory flag is read in this loop: a generic shared load
          // issued behind in-flight tcgen05.mma stalls the issuing thread
          // (measured: ~2.5x slower MMA issue).  A stalled peer shows up as
          // a timed-out barrier wait instead.
          // the stage's operands have landed and its scales are in bank s
          if (!mbar_wait_bounded(&full[s], phase, a.status) ||
              !mbar_wait_bounded(&sff[s], phase, a.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t off = (uint64_t)(s * (STAGE_BYTES >> 4));
          const uint64_t dA = dA0 + off, dB = dB0 + off;
          const uint32_t sf0 = tmem + TMEM_SF + 48u * s;
          const uint32_t acc0 = ks != k0 ? 1u : 0u;
          const int nk = (ks + 1 < n_ks || a.K % BK == 0) ? KSTEPS : (a.K - ks * BK) / MMA_K;
          if (nk == KSTEPS) {
#pragma unroll
            for (int kk = 0; kk < KSTEPS; ++kk)
              // K step kk: +32 bytes inside the 128-byte swizzle atom (+2 units)
              tc_mma(tmem + TMEM_D, dA + 2u * kk, dB + 2u * kk, kIdesc, sf0 + 12u * kk,
                     sf0 + 12u * kk + 4, kk ? 1u : acc0);
          } else {
            for (int kk = 0; kk < nk; ++kk)
              tc_mma(tmem + TMEM_D, dA + 2u * kk, dB + 2u * kk, kIdesc, sf0 + 12u * kk,
                     sf0 + 12u * kk + 4, kk ? 1u : acc0);
          }
          tc_commit(&empty[s]);  // stage free once these MMAs complete
          if (++s == NSTAGE) {
            s = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(accf);  // tile accumulated
      }
      if (!ok) *abort_flag = 1;
      // Every issued MMA completes before tensor memory is freed, whether or
      // not the epilogue waited for them (it stops early after an abort).
      tc_commit(drain);
      mbar_wait_bounded(drain, 0u, a.status);
    }
  } else if (warp >= kScaleWarp0) {
    // ------------------------------ block scales -> tensor memory
    // Warp w fills the scale columns of its tensor-memory lane quarter
    // q = w % 4 (lanes 32 q .. 32 q + 31) with tcgen05.st: for K step t and
    // operand block g (0: the X rows; 1, 2: W rows 0..127, 128..255) the
    // 4-column group the MMA reads gets, in lane 32 q + i, the 16-byte line i
    // of that block's scale atom -- what a tcgen05.cp 32x128b.warpx4 of the
    // atom writes, without occupying the tensor pipe, which then runs MMAs
    // only.  The bank of stage s is free once the stage's previous MMAs
    // completed, which the producer waited for before refilling the stage.
    const int q = warp & 3;
    const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16) + TMEM_SF;
    uint32_t s = 0, phase = 0;
    bool ok = true;
    for (int jj = 0; ok && jj < sch.n_seg; ++jj) {
      int t, k0, k1;
      sch.seg(jj, t, k0, k1);
      for (int ks = k0; ks < k1; ++ks) {
        if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(&full[s], phase, a.status))) {
          ok = false;
          break;
        }
        const uint8_t *st = smem + (size_t)s * STAGE_BYTES;
        const uint32_t col = tq + 48u * s;
#pragma unroll
        for (int kk = 0; kk < KSTEPS; ++kk) {
#pragma unroll
          for (int g = 0; g < 3; ++g) {
            const uint8_t *atom = (g == 0 ? st + OFF_SFA : st + OFF_SFB + 2048 * (g - 1)) + 512 * kk;
            tc_st4(col + 12u * kk + 4u * g, *reinterpret_cast<const uint4 *>(atom + 16 * lane));
          }
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sff[s]);
        if (++s == NSTAGE) {
          s = 0;
          phase ^= 1u;
        }
      }
    }
  } else {
    // ------------------------------ epilogue: warps 2..9
    const int quarter = warp & 3;  // tensor-memory lanes 32*quarter .. +31
    const int row_in_tile = quarter * 32 + lane;
    const int col0 = (warp - 2) / 4 * kEpiCols;  // warps 2..5: columns 0..127, 6..9: 128..255
    const float scale = (*a.s_x) * (*a.s_w);
    // bf16 of 32 fp32 values (times s_x s_w) to columns c .. c + 31 of this
    // thread's part of row m
    auto store_bf16 = [&](int64_t m, int n0, int c, const float (&v)[32], float sc) {
      if (m >= a.M) return;
      uint32_t p[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) p[i] = pack_bf16(v[2 * i] * sc, v[2 * i + 1] * sc);
      uint16_t *dst = a.y + m * a.ldy + n0 + c;
      if (n0 + c + 32 <= a.N) {
        uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
        for (int i = 0; i < 4; ++i) d4[i] = make_uint4(p[4 * i], p[4 * i + 1], p[4 * i + 2], p[4 * i + 3]);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          if (n0 + c + 2 * i < a.N) dst[2 * i] = (uint16_t)(p[i] & 0xFFFFu);
          if (n0 + c + 2 * i + 1 < a.N) dst[2 * i + 1] = (uint16_t)(p[i] >> 16);
        }
      }
    };
    int n_split = 0;
    for (int jj = 0; jj < sch.n_seg; ++jj) {
      const bool ready =
          __all_sync(0xFFFFFFFFu, mbar_wait_bounded(accf, (uint32_t)(jj & 1), a.status));
      if (!ready || *abort_flag) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      int t, k0, k1;
      sch.seg(jj, t, k0, k1);
      const int mb = t % MB, nb = t / MB;
      const int64_t m = (int64_t)mb * BM + row_in_tile;
      if (swiglu) {
        // This warp's 64 of the tile's 128 output columns: gate accumulators
        // in columns c, up in 128 + c of its lane quarter.
        const int h0 = (warp - 2) / 4 * 64;
        const uint32_t tq = tmem + ((uint32_t)(quarter * 32) << 16) + TMEM_D;
        const float sg = (*a.s_x) * (*a.s_w), su = (*a.s_x) * (*a.s_w2);
        const int n0 = nb * (BN / 2) + h0;
        uint32_t hmax = 0;
        bool finite = true;
        // h of both 32-column chunks as bf16 in registers; the accumulator
        // is handed back once the second chunk is read, before the stores
        uint32_t hp[2][16];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t rg[32], ru[32];
          tc_ld32(tq + h0 + 32 * h, rg);
          tc_ld32(tq + BN / 2 + h0 + 32 * h, ru);
          if (h == 1) {
            tc_fence_before();
            mbar_arrive(acce);
          }
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float g0 = __uint_as_float(rg[i]) * sg, u0 = __uint_as_float(ru[i]) * su;
            const float g1 = __uint_as_float(rg[i + 1]) * sg, u1 = __uint_as_float(ru[i + 1]) * su;
            hp[h][i / 2] = pack_bf16(g0 / (1.0f + expf(-g0)) * u0,   // silu(g) * u
                                     g1 / (1.0f + expf(-g1)) * u1);
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const uint32_t hb = (e ? hp[h][i / 2] >> 16 : hp[h][i / 2]) & 0x7FFFu;
              if (m < a.M && n0 + 32 * h + i + e < a.N) {
                hmax = max(hmax, hb < 0x7F80u ? hb : 0u);
                finite = finite && hb < 0x7F80u;
              }
            }
          }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) store_packed_bf16(a, m, n0 + 32 * h, hp[h]);
        for (int o = 16; o; o >>= 1) hmax = max(hmax, __shfl_xor_sync(0xFFFFFFFFu, hmax, o));
        if (!__all_sync(0xFFFFFFFFu, finite) && lane == 0) report(a.status, IMP_DEV_NONFINITE_INPUT);
        if (lane == 0 && hmax) atomicMax(a.h_amax, hmax);
        continue;
      }
      const int n0 = nb * BN + col0;
      const uint32_t tacc = tmem + ((uint32_t)(quarter * 32) << 16) + TMEM_D + col0;
      if (k0 == 0 && k1 == n_ks) {
        // Whole tile: this warp's 128 accumulator columns as bf16 in
        // registers, the accumulator handed back, then the stores (rows of
        // 64 bytes, one per lane: they take longer than the reads and now
        // run under the next tile's MMAs).
        uint32_t pk[kEpiCols / 32][16];
#pragma unroll
        for (int c = 0; c < kEpiCols / 32; ++c) {
          uint32_t r[32];
          tc_ld32(tacc + 32 * c, r);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[c][i] = pack_bf16(__uint_as_float(r[2 * i]) * scale, __uint_as_float(r[2 * i + 1]) * scale);
        }
        tc_fence_before();
        mbar_arrive(acce);  // accumulator may be overwritten now
#pragma unroll
        for (int c = 0; c < kEpiCols / 32; ++c) store_packed_bf16(a, m, n0 + 32 * c, pk[c]);
        continue;
      }
      // Split tile (stream-K): this CTA's fp32 partial of the tile goes to its
      // slot in the workspace; the last of the tile's CTAs to finish adds all
      // partials in K order (CTA order) and writes Y.
      const int sl = sch.natural(jj) == 0 ? 0 : 1;
      auto part_row = [&](int cc, int slot) {
        return a.part + ((size_t)(2 * cc + slot) * BM + row_in_tile) * BN + col0;
      };
      {
        float *pr = part_row((int)blockIdx.x, sl);
#pragma unroll
        for (int c = 0; c < kEpiCols; c += 32) {
          uint32_t r[32];
          tc_ld32(tacc + c, r);
          float4 *p4 = reinterpret_cast<float4 *>(pr + c);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            p4[i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
        }
      }
      tc_fence_before();
      mbar_arrive(acce);
      // The warps report in (CTA scope); one thread makes the CTA's stores
      // visible device-wide (a cumulative fence) and counts the segment.
      const int64_t u0 = (int64_t)t * n_ks;
      const int c_first = sch.owner(u0), c_last = sch.owner(u0 + n_ks - 1);
      __syncwarp();
      if (lane == 0) mbar_arrive(part_done);
      const uint32_t par = (uint32_t)(n_split & 1);
      ++n_split;
      if (warp == 2 && lane == 0) {
        const bool got = mbar_wait_bounded(part_done, par, a.status);
        __threadfence();
        *last_flag = got && count_split_segment(a.cnt + t, a.epoch, c_last - c_first + 1);
        __threadfence();
        mbar_arrive(flag_ready);
      }
      if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(flag_ready, par, a.status))) {
        *abort_flag = 1;
        break;
      }
      if (!*last_flag) continue;
      __threadfence();
#pragma unroll 1
      for (int c = 0; c < kEpiCols; c += 32) {
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0.0f;
        for (int cc = c_first; cc <= c_last; ++cc) {
          const float4 *q4 = reinterpret_cast<const float4 *>(part_row(cc, sch.slot_of(cc, t)) + c);
          float4 q[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) q[i] = __ldcg(q4 + i);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            v[4 * i] += q[i].x;
            v[4 * i + 1] += q[i].y;
            v[4 * i + 2] += q[i].z;
            v[4 * i + 3] += q[i].w;
          }
        }
        store_bf16(m, n0, c, v, scale);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(TMEM_COLS)
                 : "memory");
  }
}

}  // namespace

bool make_tmap_u8_2d(CUtensorMap *map, const void *base, uint64_t rows, uint64_t row_bytes,
                     uint64_t pitch, uint32_t box_rows, uint32_t box_bytes, bool swizzle128) {
  // looked up once (thread-safe static initialisation)
  static const PFN_cuTensorMapEncodeTiled_v12000 encode = []() {
    cudaDriverEntryPointQueryResult q;
    void *fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      fn = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }();
  if (!encode) return false;
  const cuuint64_t dims[2] = {row_bytes, rows};
  const cuuint64_t strides[1] = {pitch};
  const cuuint32_t box[2] = {box_bytes, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims,
                            strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

size_t gemm_mxf4_smem_bytes() { return kSmemBytes; }

namespace {
// CTAs of a launch: one per SM, at most 256 (the partial-tile slots of the
// workspace are sized for that many), at most one per unit of work.
int64_t gemm_grid(int64_t M, int64_t N, int64_t K, bool stream_k) {
  const int64_t tiles = ceil_div(M, BM) * ceil_div(N, BN);
  const int64_t units = stream_k ? tiles * ceil_div(K, BK) : tiles;
  int64_t grid = num_sms();
  if (grid > 256) grid = 256;
  return grid < units ? grid : units;
}
struct GemmWs {
  size_t cnt, part, total;
};
GemmWs gemm_ws(int64_t M, int64_t N, int64_t K) {
  GemmWs w;
  const int64_t tiles = ceil_div(M, BM) * ceil_div(N, BN);
  w.cnt = 0;
  w.part = (size_t)ceil_div(tiles * 16, 256) * 256;
  w.total = w.part + (size_t)gemm_grid(M, N, K, true) * 2 * BM * BN * sizeof(float);
  return w;
}
}  // namespace

size_t gemm_mxf4_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  if (M < 1 || N < 1 || K < 64) return 0;
  return gemm_ws(M, N, K).total;
}

struct GemmMxf4Plan::Impl {
  CUtensorMap tmA, tmB;
  GemmArgs a;
  int grid;
};
GemmMxf4Plan::GemmMxf4Plan() : impl(new Impl()) {}
GemmMxf4Plan::~GemmMxf4Plan() { delete impl; }

cudaError_t plan_gemm_mxf4(const uint8_t *x_codes, const uint8_t *x_mma_scales, const float *s_x,
                           const uint8_t *w_codes, bool w_tiled, const uint8_t *w_mma_scales,
                           const float *s_w, int64_t M, int64_t N, int64_t K, uint16_t *y,
                           int64_t ldy, int32_t *status, void *workspace, GemmMxf4Plan &plan) {
  GemmMxf4Plan::Impl &p = *plan.impl;
  memset(&p.tmA, 0, sizeof(p.tmA));
  memset(&p.tmB, 0, sizeof(p.tmB));  // not read with tiled W codes
  if (!make_tmap_u8_2d(&p.tmA, x_codes, (uint64_t)M, (uint64_t)(K / 2), (uint64_t)(K / 2), BM,
                       128, true) ||
      (!w_tiled && !make_tmap_u8_2d(&p.tmB, w_codes, (uint64_t)N, (uint64_t)(K / 2),
                                    (uint64_t)(K / 2), BN, 128, true)))
    return cudaErrorInvalidValue;
  GemmArgs &a = p.a;
  a = GemmArgs{};
  a.sfa = x_mma_scales;
  a.sfb = w_mma_scales;
  a.w_tiles = w_tiled ? w_codes : nullptr;
  a.s_x = s_x;
  a.s_w = s_w;
  a.y = y;
  a.ldy = ldy;
  a.M = (int)M;
  a.N = (int)N;
  a.K = (int)K;
  a.status = status;
  a.stream_k = workspace != nullptr;
  a.cnt = nullptr;
  a.part = nullptr;
  a.epoch = 0;
  if (workspace) {
    const GemmWs L = gemm_ws(M, N, K);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    a.cnt = reinterpret_cast<unsigned __int128 *>(ws + L.cnt);
    a.part = reinterpret_cast<float *>(ws + L.part);
    a.epoch = next_launch_epoch();
  }
  p.grid = (int)gemm_grid(M, N, K, workspace != nullptr);
  return cudaFuncSetAttribute(gemm_mxf4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)kSmemBytes);
}

cudaError_t plan_gemm_mxf4_swiglu(const uint8_t *x_codes, const uint8_t *x_mma_scales,
                                  const float *s_x, const uint8_t *gate_tiles,
                                  const uint8_t *gate_scales, const float *s_gate,
                                  const uint8_t *up_tiles, const uint8_t *up_scales,
                                  const float *s_up, int64_t M, int64_t N, int64_t K, uint16_t *h,
                                  int64_t ldh, uint32_t *h_amax, int32_t *status,
                                  GemmMxf4Plan &plan) {
  const cudaError_t e = plan_gemm_mxf4(x_codes, x_mma_scales, s_x, gate_tiles, true, gate_scales,
                                       s_gate, M, N, K, h, ldh, status, nullptr, plan);
  if (e != cudaSuccess) return e;
  GemmArgs &a = plan.impl->a;
  a.w2_tiles = up_tiles;
  a.sfb2 = up_scales;
  a.s_w2 = s_up;
  a.h_amax = h_amax;
  plan.impl->grid = (int)gemm_grid(M, 2 * N, K, false);  // 128 output columns per tile
  return cudaSuccess;
}

cudaError_t enqueue_gemm_mxf4(const GemmMxf4Plan &plan, cudaStream_t stream) {
  const GemmMxf4Plan::Impl &p = *plan.impl;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_mxf4_kernel, p.tmA, p.tmB, p.a);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace impfp4
