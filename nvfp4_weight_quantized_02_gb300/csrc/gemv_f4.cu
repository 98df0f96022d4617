// Decode GEMV (M <= 16) with the NVFP4 weight fed straight to the
// block-scaled FP4 tensor cores:
//   y[m][n] = s_w * sum_k x[m][k] * e2m1(c[n][k]) * e4m3(sb[n][k/16]).
//
// Decode is bandwidth-bound (imp README, "How it works"; "1. The big
// picture", section "The most important number in this book"), so the aim
// is to move W from HBM into the tensor cores with no per-weight work on the
// CUDA cores at all.  tcgen05.mma.kind::mxf4nvf4 multiplies E2M1 codes with
// E4M3 scales per 16 elements on both operands, exactly the weight format.
// X, in bf16, is not: it is rewritten per call as a short sum of NVFP4
// "components" (one extra operand row per component), the MMA's B operand:
//
//   x * 2^sh = sum_{c < 8} 2^(4 - 2c) * e4m3(sb_c[b]) * e2m1(q_c[k]),
//
// with the power-of-two prescale 2^sh putting the row's max|x| in
// [2^14, 2^15) and component c quantizing the residual left by components
// 0..c-1 (block amax / 6 -> E4M3 scale; value / scale -> E2M1, nearest).
// Each component shrinks a block's residual by a factor of at least ~5.6,
// so eight of them leave a few 1e-9 of the block's largest |x| at most (fp32
// rounding of the residual updates dominates).  Every MMA product
// (E2M1 x E4M3 x E2M1 x E4M3) is exact; accumulation is fp32 in tensor
// memory.  y sums the component columns with their power-of-two weights, in
// a fixed order.
//
// Work split over the (128-row tile, 256-element K chunk) grid, one CTA per
// SM at most:
//  * whole tiles, as evenly as they divide (at least 3/4 as many tiles as
//    SMs);
//  * fewer tiles: each tile's K chunks split over a thread-block cluster of
//    S CTAs, whose fp32 partial sums meet in rank 0's shared memory
//    (distributed shared memory) and are added in rank (= K) order;
//  * otherwise stream-K: the tile-major chunk sequence cut into equal
//    contiguous ranges; a partial tile's CTAs leave fp32 partial sums in the
//    workspace and the last of them to finish adds them in K order.
//
// Two kernels share those schedules:
//  * gemv_f4r_kernel (M <= 2, the usual decode case): X's components are
//    held in shared memory for the whole call (B "slots", one per K chunk
//    the CTA sees).  Warp 4 streams W through an 8-deep ring (a weight in the
//    tensor-core layout of quantize.cuh: two contiguous bulk copies per
//    stage; row-major: 2-D TMA of 128 x 128-byte code tiles, 128-byte
//    swizzle, and 128 x 16-byte scale rows, which warp 6 relays into atoms)
//    and never waits for the previous kernel (W is never written on the
//    stream).  The slots come from a split kernel (xsplit_slots_kernel, once
//    per call; warp 5 copies them in) or, with at most six chunks per CTA,
//    from the kernel's own warps 5, 7 and 8..11, one slot each.  Warps 0..3
//    issue the MMAs (stage i -> issuer i % 4), warps 8..11 run the epilogue.
//    The same kernel serves FP8-E4M3 weights (kind::f8f6f4, X split into
//    E4M3 components by xsplit_f8_kernel, no block scales).
//  * gemv_f4_kernel (any M <= 16, one pass over W): a separate split
//    kernel (xsplit_kernel) writes the components and scale atoms to the
//    workspace, and they travel with W in each stage of the ring; producer
//    warp 4, epilogue warps 8..11, and MMA issuers from warp 0 -- four for
//    B operands of 16 or 32 rows (8-deep ring), two for 64 (6-deep), one for
//    128 (5-deep): a wider MMA takes longer, so fewer issuers keep ahead of
//    HBM, and the wider B stages fill the shared memory sooner.
//  * gemv_f4c_kernel (M <= 2, several calls in one launch): the resident
//    kernel's roles run call after call through one ring; each CTA splits
//    its chunks of a call's X itself (warps 5..11), after a per-call count
//    of finished CTAs when X is the previous call's output.
// Issuer: one thread copies both operands' scale atoms of a stage to tensor
// memory (tcgen05.cp) and issues four M=128 x N=N_MMA x K=64 MMAs into its
// own accumulator.  One issuing thread sustains one MMA per ~130 cycles;
// three or four keep the tensor core ahead of HBM.  Epilogue: thread = tile
// row (its tensor-memory lane).
// Every wait is bounded; on a timeout the kernel reports IMP_DEV_TIMEOUT,
// drains its own copies and MMAs, frees tensor memory and returns.
#include <atomic>
#include <cstring>
#include <chrono>
#include <mutex>
#include <random>

#include "gemv.cuh"
#include "tma.cuh"

namespace impfp4 {

namespace {

constexpr int kNC = 8;          // components per row of X
constexpr int kTileRows = 128;
constexpr int kChunkK = 256;    // K per stage (four K64 MMAs)
constexpr uint32_t kTmemCols = 512;
constexpr int kXsplitThreads = 256;
constexpr int kPrefetch = 12;   // stages of W prefetched into L2 at the start
constexpr int kEpiWarp0 = 8;    // warps 8..11: epilogue (tensor-memory lane quarters 0..3)
constexpr int kRelayWarp = 6;   // row-major W: relays the scale rows into atoms
constexpr int kThreads = 384;
// The split-tile partials are sized for at most kMaxGrid CTAs, so the
// workspace size does not depend on the device.
constexpr int kMaxGrid = 256;

constexpr int kMaxRowsX = 16;  // rows of X per launch (operand rows: 8 per row)

// ---- streamed-B kernel
constexpr int kProducerS = 4;
// Issuers and ring depth per operand width: the accumulators (two per
// issuer, N_MMA columns each) and the scale banks (32 columns per ring slot)
// share the 512 tensor-memory columns, and the ring fills the shared memory.
// A wider B makes each MMA slower, so fewer issuers keep up with HBM.
template <int NMMA> struct CfgS;
template <> struct CfgS<16> { static constexpr int NI = 4, NS = 8; };
template <> struct CfgS<32> { static constexpr int NI = 4, NS = 8; };
template <> struct CfgS<64> { static constexpr int NI = 2, NS = 6; };
template <> struct CfgS<128> { static constexpr int NI = 1, NS = 5; };
template <int NMMA> struct StageS {
  static constexpr uint32_t W = 0;                 // 128 x 128 B, swizzled
  static constexpr uint32_t B = 16384;             // NMMA x 128 B, swizzled
  static constexpr uint32_t RAW = B + 128 * NMMA;  // W scales, 128 x 16 B
  static constexpr uint32_t SFA = RAW + 2048;      // 4 atoms
  static constexpr uint32_t SFB = SFA + 2048;      // 4 atoms
  static constexpr uint32_t BYTES = SFB + 2048;    // multiple of 1024
  static constexpr uint32_t TX = 16384 + 128 * NMMA + 2048 + 2048;
};

// ---- resident-B kernel (M <= 2, N_MMA = 16)
constexpr int kIssuersR = 4, kProducerR = 4, kNSR = 8;  // a multiple of the issuers: stage st and st - 8, same issuer
constexpr int kLoaderWarpR = 5;                          // warp 5: copies the B slots in (FP8)
constexpr int kSplitWarpX = 7;                           // warps 5, 7, 8..11 split X (NVFP4)
constexpr int kSplitW = 6;                               // split warps, one slot each
constexpr int kSplitWarps = 8;                           // chunks per CTA of the split kernel
// Weight formats of the resident kernel: NVFP4 (E2M1 codes, E4M3 block
// scales; X split into NVFP4 components; tcgen05.mma kind::mxf4nvf4) and
// FP8 E4M3 with one tensor scale (X split into E4M3 components; kind::f8f6f4,
// no block scales).  A stage is 128 rows x 128 bytes of W either way: 256
// elements of NVFP4 or 128 of FP8.
enum { kFmtNv = 0, kFmtF8 = 1 };
template <int FMT> struct FmtR;
template <> struct FmtR<kFmtNv> {
  static constexpr int kChunk = 256;          // K elements per stage
  static constexpr uint32_t kStageBytes = 18432, kTX = 16384 + 2048;
  static constexpr uint32_t kSlotSf = 1024;   // B scale bytes per slot
  static constexpr int kMaxSlots = 24;
};
template <> struct FmtR<kFmtF8> {
  static constexpr int kChunk = 128;
  static constexpr uint32_t kStageBytes = 16384, kTX = 16384;
  static constexpr uint32_t kSlotSf = 0;
  static constexpr int kMaxSlots = 40;
};
// W scales land where their atoms go: a row-major weight's 128 x 16-byte
// scale rows are relaid in place (read, warp sync, write).
template <int FMT> struct StageRT {
  static constexpr uint32_t W = 0, RAW = 16384, SFA = 16384, BYTES = FmtR<FMT>::kStageBytes;
  static constexpr uint32_t TX = FmtR<FMT>::kTX;
};
using StageR = StageRT<kFmtNv>;
// B slot image of one K chunk (written into shared memory by the resident
// kernel's split warps, split_chunk_slot): codes, 2 KB = 16
// operand rows x 128 B, row n at 128 n with its 16-byte unit u at unit
// u ^ (n % 8) (the 128-byte swizzle); scales, 1 KB = four K64 steps of 256 B,
// operand row n of step t at 256 t + 16 n (the row's 4 block scales; 12 zero
// bytes): lines 0..15 of a 512-byte atom, whose copy reads 256 bytes past
// them (the next step's lines, or a zeroed pad) into lanes no N = 16 MMA
// reads.  Operand row 8 m + c holds component c of row m of X; rows past the
// last component are zero.

// A call multiplies one X by up to kMaxGroups weights of the same K (for
// example a layer's q, k and v projections): their 128-row tiles follow each
// other in the call's tile sequence, group g from tile tile0 on, and each
// keeps its own tensor scale and output.  An ordinary call has one group.
constexpr int kMaxGroups = 4;
struct F4Group {
  const uint8_t *wc;    // prepared weight: code tiles [128-row block][chunk][16 KB]
  const uint8_t *wsa;   // prepared weight: scale atoms [128-row block][K/64][512 B]
  const float *ts;      // tensor scale s_w
  uint16_t *y;          // bf16[M][ldy]
  int64_t N, ldy;
  int tile0;            // the group's first tile in the call
};

struct F4Args {
  const uint16_t *x;    // resident kernel: X rows
  int64_t ldx;
  int M;
  int64_t K;
  const uint8_t *sfb;   // X component scales: streamed kernel atoms [K/64][512]; resident kernel slot images [K/256][1 KB]
  const uint8_t *slot_codes;  // resident kernel: X component codes, slot images [K/256][2 KB]
  const int32_t *sh;    // streamed kernel: per-row prescale exponents
  float *part;          // split-tile partial sums, [CTA][first/last segment][128][N_MMA / 8]
  unsigned __int128 *cnt;   // per tile: epoch, its check word and segments finished
  int32_t *status;
  int n_tiles;
  int n_chunks;         // K / 256
  unsigned long long epoch;  // unique per launch
  int n_slots;          // resident kernel: B slots in shared memory
  int sched;            // kSchedStreamK / kSchedWhole / kSchedCluster
  int ksplit;           // kSchedCluster: CTAs per tile (the cluster size)
  int grid;             // CTAs the call is spread over (0: the whole grid)
  unsigned int *cnt32;  // per tile: segments finished, cleared before the launch counts
                        // (a persistent launch's own protocol); nullptr: cnt
  const uint16_t *x2;   // chained calls: X = bf16(silu(x) * x2) when set
  int64_t ldx2;
  int n_groups;         // weights of the call (row-major weight: 1)
  F4Group grp[kMaxGroups];
};

// Group of call tile `tile` (groups in tile order).
__device__ __forceinline__ int group_of(const F4Args &a, int tile) {
  int g = 0;
#pragma unroll
  for (int i = 1; i < kMaxGroups; ++i) g += (i < a.n_groups && tile >= a.grp[i].tile0) ? 1 : 0;
  return g;
}
// a.grp[g] without a dynamically indexed parameter access
__device__ __forceinline__ F4Group group_at(const F4Args &a, int g) {
  F4Group r = a.grp[0];
#pragma unroll
  for (int i = 1; i < kMaxGroups; ++i)
    if (g == i) r = a.grp[i];
  return r;
}
// Code tiles and scale atoms of one call tile of a prepared weight (chunk ch
// at wc + 16 KB ch and wsa + 2 KB ch), looked up again only when the tile
// changes: the producer's per-stage work stays a few adds.
struct PreparedTile {
  int tile = -1;
  const uint8_t *wc = nullptr, *wsa = nullptr;
  __device__ __forceinline__ void at(const F4Args &a, int t, int nch) {
    if (t == tile) return;
    const F4Group g = group_at(a, group_of(a, t));
    const int64_t lt = t - g.tile0;
    wc = g.wc + lt * nch * 16384;
    wsa = g.wsa + lt * (a.K / 64) * 512;
    tile = t;
  }
};

struct F4Bars {
  uint64_t full[8], empty[8], sf_ready[8];
  uint64_t d_full[4][2], d_empty[2];
  uint64_t drain[4];
  uint64_t part_done, flag_ready;  // split-tile hand-off among the epilogue warps
  uint64_t cl_full;                // kSchedCluster, rank 0: the other ranks' partials arrived
  uint64_t b_ready;                // resident kernel: every B slot has landed (copied in)
  uint32_t tmem;
  int last;
};
// Resident kernel splitting X itself: a barrier per B slot and the split
// warps' per-row maxima (after the cluster reduction buffer).
struct F4SplitBars {
  uint64_t slot_ready[6];
  uint32_t xmax[6][2];
};

__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                          uint32_t layout) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version
  d |= (uint64_t)(layout & 7u) << 61;
  return d;
}
constexpr uint32_t kSw128 = 2, kNoSwizzle = 0;

template <int NMMA>
__host__ __device__ constexpr uint32_t idesc_f4() {
  // kind::mxf4nvf4: A and B E2M1 (format 1), K-major, N >> 3 at bit 17, M >> 4 at bit 24
  return (1u << 7) | (1u << 10) | ((uint32_t)(NMMA >> 3) << 17) |
         ((uint32_t)(kTileRows >> 4) << 24);
}

template <int NMMA>
__host__ __device__ constexpr uint32_t idesc_f8() {
  // kind::f8f6f4: D fp32 (1 at bit 4), A and B E4M3 (format 0), K-major,
  // N >> 3 at bit 17, M >> 4 at bit 24
  return (1u << 4) | ((uint32_t)(NMMA >> 3) << 17) | ((uint32_t)(kTileRows >> 4) << 24);
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void tc_cp_sf(uint32_t taddr, uint64_t sdesc_) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc_)
               : "memory");
}
__device__ __forceinline__ void tc_mma_f4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, "
      "[%5], [%6], p;\n}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb)
      : "memory");
}
__device__ __forceinline__ void tc_mma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void tc_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t *slot) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(slot)),
               "r"(kTmemCols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_free(uint32_t tmem) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
               : "memory");
}

__device__ __forceinline__ float e4m3_to_f32(uint32_t b) { return f16lo_to_f32(e4m3x2_to_f16x2(b)); }

// ---- thread-block cluster helpers (kSchedCluster) -----------------------------

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// The address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_map(uint32_t saddr, uint32_t rank) {
  uint32_t d;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(saddr), "r"(rank));
  return d;
}
__device__ __forceinline__ void st_cluster_f32(uint32_t caddr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(caddr), "f"(v) : "memory");
}
__device__ __forceinline__ void mbar_arrive_remote(uint32_t caddr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(caddr) : "memory");
}
// Bounded wait on a local mbarrier whose arrivals come from other CTAs of the
// cluster (acquire at cluster scope: their stores before the arrive are seen).
__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint64_t *bar, uint32_t parity,
                                                          int32_t *status) {
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    for (int i = 0; i < 64; ++i) {
      uint32_t ok;
      asm volatile(
          "{\n.reg .pred p;\nmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
          "selp.u32 %0, 1, 0, p;\n}"
          : "=r"(ok)
          : "r"(smem_u32(bar)), "r"(parity)
          : "memory");
      if (ok) return true;
    }
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      report(status, IMP_DEV_TIMEOUT);
      return false;
    }
  }
}
// Every thread of every CTA of the cluster (release / acquire).
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;\nbarrier.cluster.wait.acquire;" ::: "memory");
}

// ---- the split of X ----------------------------------------------------------

// Power-of-two prescale putting max|x| (bf16 bits of the magnitude) in
// [2^14, 2^15); 0 for an all-zero or non-finite row.
__device__ __forceinline__ int prescale_exponent(uint32_t mx_bits16) {
  const float xmax = __uint_as_float(mx_bits16 << 16);
  if (!(xmax > 0.0f && xmax < __int_as_float(0x7F800000))) return 0;
  int e;
  frexpf(xmax, &e);
  return 15 - e;
}

// h = silu(g) * u for eight bf16 pairs, in fp32 (silu(v) = v / (1 + e^-v),
// as the prefill SwiGLU epilogue evaluates it), rounded to bf16: the X of a
// down projection whose input is the activation of its gate and up outputs.
__device__ __forceinline__ uint32_t swiglu_bf16x2(uint32_t g2, uint32_t u2) {
  const float g0 = __uint_as_float(g2 << 16), g1 = __uint_as_float(g2 & 0xFFFF0000u);
  const float u0 = __uint_as_float(u2 << 16), u1 = __uint_as_float(u2 & 0xFFFF0000u);
  const float h0 = g0 / (1.0f + expf(-g0)) * u0, h1 = g1 / (1.0f + expf(-g1)) * u1;
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(h0)) |
         (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(h1)) << 16;
}
__device__ __forceinline__ uint4 swiglu_bf16x8(const uint4 g, const uint4 u) {
  return make_uint4(swiglu_bf16x2(g.x, u.x), swiglu_bf16x2(g.y, u.y), swiglu_bf16x2(g.z, u.z),
                    swiglu_bf16x2(g.w, u.w));
}

__device__ __forceinline__ uint32_t absmax_bf16x8(const uint4 v) {
  return max(max(max(v.x & 0x7FFFu, v.x >> 16 & 0x7FFFu), max(v.y & 0x7FFFu, v.y >> 16 & 0x7FFFu)),
             max(max(v.z & 0x7FFFu, v.z >> 16 & 0x7FFFu), max(v.w & 0x7FFFu, v.w >> 16 & 0x7FFFu)));
}

// One 16-element block of X (16 bf16 in v, element order) -> eight
// components: code[c] = 16 E2M1 codes (element 2i in the low nibble of byte
// i), sb[c] = the E4M3 block scale in units of 2^(4 - 2c).
__device__ __forceinline__ float pow2f(int e) {  // 2^e, -126 <= e <= 127
  return __int_as_float((127 + e) << 23);
}

__device__ __forceinline__ void split_block_regs(const uint4 (&v)[2], int sh, uint2 (&code)[kNC],
                                                 uint32_t (&sb)[kNC]) {
  // x * 2^sh as two exact power-of-two products (|sh| may exceed 127)
  const float p1 = pow2f(sh / 2), p2 = pow2f(sh - sh / 2);
  float r[16];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t w[4] = {v[h].x, v[h].y, v[h].z, v[h].w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      r[8 * h + 2 * t] = bf16_bits_to_f32(w[t] & 0xFFFFu) * p1 * p2;
      r[8 * h + 2 * t + 1] = bf16_bits_to_f32(w[t] >> 16) * p1 * p2;
    }
  }
#pragma unroll
  for (int c = 0; c < kNC; ++c) {
    float m8[8];  // |r| max as a tree
#pragma unroll
    for (int k = 0; k < 8; ++k) m8[k] = fmaxf(fabsf(r[k]), fabsf(r[k + 8]));
#pragma unroll
    for (int k = 0; k < 4; ++k) m8[k] = fmaxf(m8[k], m8[k + 4]);
    const float amax = fmaxf(fmaxf(m8[0], m8[2]), fmaxf(m8[1], m8[3]));
    // Any scale is valid -- the residual tracks what was taken -- so a
    // reciprocal stands in for the divisions.
    sb[c] = f32_to_e4m3_satfinite(amax * (1.0f / 6.0f) * pow2f(2 * c - 4));
    const float d = e4m3_to_f32(sb[c]) * pow2f(4 - 2 * c);
    uint32_t cw[2] = {0u, 0u};
    if (d > 0.0f) {
      const float inv = 1.0f / d;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float q[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) q[k] = r[8 * h + k] * inv;
        cw[h] = f32x8_to_e2m1_packed(q);
        uint32_t e[4];
        e2m1x8_to_f16x2x4(cw[h], e);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          // e2m1 * d is exact in fp32; one rounding in the subtraction
          r[8 * h + 2 * t] = fmaf(-f16lo_to_f32(e[t]), d, r[8 * h + 2 * t]);
          r[8 * h + 2 * t + 1] = fmaf(-f16hi_to_f32(e[t]), d, r[8 * h + 2 * t + 1]);
        }
      }
    }
    code[c] = make_uint2(cw[0], cw[1]);
  }
}

// The same for a block read from p (bf16, 16-byte aligned).
__device__ __forceinline__ void split_block(const uint16_t *p, int sh, uint2 (&code)[kNC],
                                            uint32_t (&sb)[kNC]) {
  const uint4 v[2] = {__ldg(reinterpret_cast<const uint4 *>(p)),
                      __ldg(reinterpret_cast<const uint4 *>(p) + 1)};
  split_block_regs(v, sh, code, sb);
}

// ---- stream-K bookkeeping -----------------------------------------------------

// Work schedules over the (128-row tile, 256-element chunk) sequence,
// tile-major; every CTA gets one contiguous range of it:
//  * kSchedStreamK: equal ranges (tiles split between CTAs are summed from
//    fp32 partials in the workspace by the tile's last CTA);
//  * kSchedWhole: whole tiles, as evenly as they divide (no split tiles);
//  * kSchedCluster: each tile's chunks split evenly over the S CTAs of one
//    thread-block cluster (CTA rank r takes part r); the ranks' partial sums
//    meet in rank 0's shared memory (distributed shared memory, no global
//    round trips) and rank 0 adds them in K order.
enum { kSchedStreamK = 0, kSchedWhole = 1, kSchedCluster = 2 };

struct StreamK {
  int64_t total, g_begin, g_end;
  int nch, n_st, n_seg, G;
  int tile0, ch0;  // tile and chunk of the CTA's first stage
  int e0, sl, nl;  // end of the first segment; start and length of the last
  // grid > 0: the call is spread over CTAs 0..grid-1 only (the others get
  // nothing), so that a stream-K call with fewer chunks than CTAs leaves no
  // empty CTA between the owners of a tile.
  __device__ StreamK(int n_tiles, int n_chunks, int sched, int S, int grid = 0) {
    G = grid > 0 ? grid : (int)gridDim.x;
    nch = n_chunks;
    total = (int64_t)n_tiles * nch;
    if ((int)blockIdx.x >= G) {
      g_begin = g_end = total;
    } else if (sched == kSchedWhole) {
      g_begin = (int64_t)n_tiles * blockIdx.x / G * nch;
      g_end = (int64_t)n_tiles * (blockIdx.x + 1) / G * nch;
    } else if (sched == kSchedCluster) {
      const int64_t t = blockIdx.x / S, r = blockIdx.x % S;
      g_begin = t * nch + nch * r / S;
      g_end = t * nch + nch * (r + 1) / S;
    } else {
      g_begin = total * blockIdx.x / G;
      g_end = total * (blockIdx.x + 1) / G;
    }
    n_st = (int)(g_end - g_begin);
    n_seg = n_st > 0 ? (int)((g_end - 1) / nch - g_begin / nch) + 1 : 0;
    tile0 = (int)(g_begin / nch);
    ch0 = (int)(g_begin % nch);
    e0 = n_seg > 0 ? seg_end(0) : 0;
    sl = n_seg > 0 ? seg_begin(n_seg - 1) : 0;
    nl = n_st - sl;
  }
  __device__ int seg_begin(int j) const {  // first stage of local segment j
    return j == 0 ? 0 : j * nch - ch0;
  }
  __device__ int seg_end(int j) const { return j + 1 < n_seg ? seg_begin(j + 1) : n_st; }
  // Processing order: the first segment, then the last, then the middle ones
  // (whole tiles), so a CTA's split tiles finish early and their fix-ups
  // overlap whole-tile work.  jj: processing position of a segment; i: of a
  // stage.
  __device__ int proc_seg(int jj) const { return jj == 0 ? 0 : jj == 1 ? n_seg - 1 : jj - 1; }
  __device__ int pbegin(int jj) const {
    if (jj == 0) return 0;
    if (jj == 1) return e0;
    return nl + seg_begin(jj - 1);
  }
  __device__ int pend(int jj) const {
    const int j = proc_seg(jj);
    return pbegin(jj) + seg_end(j) - seg_begin(j);
  }
  __device__ int stage_of(int i) const {
    if (n_seg < 2) return i;
    return i < e0 ? i : i < e0 + nl ? sl + (i - e0) : i - nl;
  }
  // tile and chunk of stage st (32-bit arithmetic)
  __device__ void tile_ch(int st, int &tile, int &ch) const {
    const int c = ch0 + st, q = c / nch;
    tile = tile0 + q;
    ch = c - q * nch;
  }
  // CTA owning global chunk g
  __device__ int owner(int64_t g) const { return (int)(((g + 1) * G - 1) / total); }
};

// ---- issuer and epilogue loops, shared by both kernels ------------------------

// W scale relay (one warp, weights in row-major layout): per stage, the
// 128 x 16-byte scale rows that landed with the codes -> four 512-byte atoms
// (the tcgen05.cp source layout), then sf_ready[s].  The issuers wait on
// sf_ready instead of full, so the relay stays off their path.
template <int NS, class Stage>
__device__ void relay_loop(uint8_t *smem, F4Bars &bars, const StreamK &sk, int lane,
                           int32_t *status) {
  for (int i = 0; i < sk.n_st; ++i) {
    const int s = i % NS;
    if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(&bars.full[s], (uint32_t)((i / NS) & 1), status)))
      return;
    uint8_t *stg = smem + (size_t)s * Stage::BYTES;
    uint4 rq[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      rq[q] = *reinterpret_cast<const uint4 *>(stg + Stage::RAW + 16 * (lane + 32 * q));
    __syncwarp();  // the atoms may overwrite the rows just read
    *reinterpret_cast<uint4 *>(stg + Stage::SFA + 0 * 512 + 16 * lane) = make_uint4(rq[0].x, rq[1].x, rq[2].x, rq[3].x);
    *reinterpret_cast<uint4 *>(stg + Stage::SFA + 1 * 512 + 16 * lane) = make_uint4(rq[0].y, rq[1].y, rq[2].y, rq[3].y);
    *reinterpret_cast<uint4 *>(stg + Stage::SFA + 2 * 512 + 16 * lane) = make_uint4(rq[0].z, rq[1].z, rq[2].z, rq[3].z);
    *reinterpret_cast<uint4 *>(stg + Stage::SFA + 3 * 512 + 16 * lane) = make_uint4(rq[0].w, rq[1].w, rq[2].w, rq[3].w);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars.sf_ready[s]);
  }
}

// Every MMA of issuer `is` completes before tensor memory is freed.
__device__ __forceinline__ void issuer_drain(F4Bars &bars, int is, int lane, int32_t *status) {
  if (lane == 0) {
    tc_commit(&bars.drain[is]);
    mbar_wait_bounded(&bars.drain[is], 0u, status);
  }
}

// Issuer `is` of NI: stages (in processing order) i = is, is + NI, ...  Lane
// 0 copies both operands' scale atoms of the stage into its bank of tensor
// memory (tcgen05.cp) and issues its four K64 MMAs into the issuer's own
// accumulator; the epilogue adds the NI accumulators.  `b_desc(i, st, t)` /
// `sfb_desc(i, st, t)`: the B operand and its scale atom for K64 step t of
// processing position i (stage st); `b_wait(st)`: waits (bounded) until that
// B is in shared memory.  All per-stage bookkeeping is 32-bit integer work:
// every instruction of this loop sits between MMA issues.
// Chained calls (one launch running several calls in turn) continue the ring
// and the accumulator hand-off: ib = ring positions and jb = segments that
// the earlier calls used; there an issuer with no stage in a segment still
// waits for the accumulator's previous segment to be read, since a run of
// such segments could otherwise complete d_full two phases ahead of the
// epilogue.  Returns false after a wait gave up.
template <int NI, int NS, int NMMA, bool PREP, class Stage, class BDesc, class SFBDesc, class BWait>
__device__ bool issuer_loop(uint8_t *smem, F4Bars &bars, uint32_t tmem, const StreamK &sk,
                            int is, int lane, int32_t *status, BDesc b_desc, SFBDesc sfb_desc,
                            BWait b_wait, int ib = 0, int jb = 0, bool chain = false) {
  constexpr uint32_t kIdesc = idesc_f4<NMMA>();
  constexpr uint32_t kSF0 = 2 * NI * NMMA;  // scale columns after the accumulators
  static_assert(kSF0 + 32 * NS <= kTmemCols, "tensor memory plan");
  // Stages i and i + NS share a ring slot; with NS a multiple of NI the same
  // issuer takes both, in order, so it never waits on a slot's full barrier
  // more than one phase ahead (a parity wait cannot tell phase p from p + 2).
  static_assert(NS % NI == 0, "ring depth must be a multiple of the issuer count");
  const uint32_t sbase = smem_u32(smem);
  const uint64_t dA0 = sdesc(sbase + Stage::W, 16, 1024, kSw128);
  const uint64_t dSA0 = sdesc(sbase + Stage::SFA, 0, 128, kNoSwizzle);
  bool ok = true;
  for (int jj = 0; jj < sk.n_seg && ok; ++jj) {
    const int p0 = sk.pbegin(jj), p1 = sk.pend(jj);
    const int J = jb + jj, d = J & 1;
    const int first = p0 + ((is - ib - p0) % NI + NI) % NI;  // this issuer's first stage
    if (chain && first >= p1 && J >= 2 &&
        !__all_sync(0xFFFFFFFFu, mbar_wait_bounded(&bars.d_empty[d], (uint32_t)((J / 2 - 1) & 1), status))) {
      ok = false;
      break;
    }
    for (int i = first; i < p1; i += NI) {
      const int s = (ib + i) % NS, st = sk.stage_of(i);
      if (i == first && J >= 2 &&
          !__all_sync(0xFFFFFFFFu, mbar_wait_bounded(&bars.d_empty[d], (uint32_t)((J / 2 - 1) & 1), status))) {
        ok = false;
        break;
      }
      // the stage's W (and, row-major, its relaid scale atoms) and its B
      uint64_t *ready = PREP ? &bars.full[s] : &bars.sf_ready[s];
      if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(ready, (uint32_t)(((ib + i) / NS) & 1), status) &&
                                       b_wait(st))) {
        ok = false;
        break;
      }
      if (lane == 0) {
        tc_fence_after();
        const uint64_t off = (uint64_t)(s * (Stage::BYTES >> 4));
        // Scale bank s (32 columns: step t's W atom at 8 t, B's at 8 t + 4):
        // its previous user, stage i - NS, completed before the producer
        // refilled slot s.
        const uint32_t sf = tmem + kSF0 + 32u * (uint32_t)s;
        const uint32_t dt = tmem + (uint32_t)((2 * is + d) * NMMA);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          tc_cp_sf(sf + 8u * t, dSA0 + off + 32u * t);
          tc_cp_sf(sf + 8u * t + 4, sfb_desc(i, st, t));
        }
#pragma unroll
        for (int t = 0; t < 4; ++t)
          tc_mma_f4(dt, dA0 + off + 2u * t, b_desc(i, st, t), kIdesc, sf + 8u * t, sf + 8u * t + 4,
                    (i == first && t == 0) ? 0u : 1u);
        tc_commit(&bars.empty[s]);
      }
      __syncwarp();
    }
    // one completion per segment, whether or not this issuer had a stage in it
    if (ok && lane == 0) tc_commit(&bars.d_full[is][d]);
    __syncwarp();
  }
  if (!chain) issuer_drain(bars, is, lane, status);
  return ok;
}

// Issuer of the FP8 weight format: the same stage order and accumulators as
// issuer_loop, four K32 MMAs (kind::f8f6f4, no block scales) per stage.
template <int NI, int NS, int NMMA, class Stage, class BDesc, class BWait>
__device__ void issuer_loop_f8(uint8_t *smem, F4Bars &bars, uint32_t tmem, const StreamK &sk,
                               int is, int lane, int32_t *status, BDesc b_desc, BWait b_wait) {
  constexpr uint32_t kIdesc = idesc_f8<NMMA>();
  static_assert(2 * NI * NMMA <= kTmemCols, "tensor memory plan");
  static_assert(NS % NI == 0, "ring depth must be a multiple of the issuer count");
  const uint64_t dA0 = sdesc(smem_u32(smem) + Stage::W, 16, 1024, kSw128);
  bool ok = true;
  for (int jj = 0; jj < sk.n_seg && ok; ++jj) {
    const int p0 = sk.pbegin(jj), p1 = sk.pend(jj);
    const int d = jj & 1;
    const int first = p0 + ((is - p0) % NI + NI) % NI;
    for (int i = first; i < p1; i += NI) {
      const int s = i % NS, st = sk.stage_of(i);
      if (i == first && jj >= 2 &&
          !__all_sync(0xFFFFFFFFu, mbar_wait_bounded(&bars.d_empty[d], (uint32_t)((jj / 2 - 1) & 1), status))) {
        ok = false;
        break;
      }
      if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(&bars.full[s], (uint32_t)((i / NS) & 1), status) &&
                                       b_wait(st))) {
        ok = false;
        break;
      }
      if (lane == 0) {
        tc_fence_after();
        const uint64_t off = (uint64_t)(s * (Stage::BYTES >> 4));
        const uint32_t dt = tmem + (uint32_t)((2 * is + d) * NMMA);
#pragma unroll
        for (int t = 0; t < 4; ++t)
          tc_mma_f8(dt, dA0 + off + 2u * t, b_desc(i, st, t), kIdesc,
                    (i == first && t == 0) ? 0u : 1u);
        tc_commit(&bars.empty[s]);
      }
      __syncwarp();
    }
    if (ok && lane == 0) tc_commit(&bars.d_full[is][d]);
    __syncwarp();
  }
  if (lane == 0) {
    tc_commit(&bars.drain[is]);
    mbar_wait_bounded(&bars.drain[is], 0u, status);
  }
}

// Epilogue warps (kEpiWarp0..+3): per segment, the NI accumulators of each
// row -> y (whole tile) or a partial sum (split tile, last CTA adds them).
// Column c of a row's operand rows carries component c mod 8 with weight
// 2^(4 - 2c) (NVFP4 components) or 2^(-4c) (E4M3 components).
// Chained calls pass the ring positions (ib) and segments (jb) of the earlier
// calls and carry the split-tile count (n_split) from call to call.
// Returns false after a wait gave up.
template <int NI, int NMMA, int FMT = kFmtNv>
__device__ bool epilogue_loop(const F4Args &a, F4Bars &bars, uint32_t tmem, const StreamK &sk,
                              int warp, int lane, const int (&sh)[kMaxRowsX], float *red,
                              int ib, int jb, int &n_split) {
  constexpr int MR = NMMA / kNC;  // rows of X the operand holds (>= M)
  const int q = warp & 3;
  const int row_in_tile = 32 * q + lane;
  float osc[kMaxGroups];  // the groups' tensor scales, loaded together
#pragma unroll
  for (int g = 0; g < kMaxGroups; ++g) osc[g] = g < a.n_groups ? *a.grp[g].ts : 0.0f;
  volatile int *last_flag = &bars.last;
  for (int jj = 0; jj < sk.n_seg; ++jj) {
    const int J = jb + jj, d = J & 1, j = sk.proc_seg(jj);
    const int s0 = sk.seg_begin(j), s1 = sk.seg_end(j);
    int T32, c0;
    sk.tile_ch(s0, T32, c0);
    const int64_t T = T32;
    const int c1 = c0 + (s1 - s0);
    bool ok = true;
    for (int i = 0; i < NI; ++i)
      ok = ok && mbar_wait_bounded(&bars.d_full[i][d], (uint32_t)((J >> 1) & 1), a.status);
    if (!__all_sync(0xFFFFFFFFu, ok)) return false;
    tc_fence_after();
    float acc[MR];
#pragma unroll
    for (int m = 0; m < MR; ++m) acc[m] = 0.0f;
    const int p0 = sk.pbegin(jj);
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      if (s1 - s0 >= NI || ((i - ib - p0) % NI + NI) % NI < s1 - s0) {  // issuer i had a stage
#pragma unroll
        for (int h = 0; h < NMMA / 16; ++h) {
          uint32_t v[16];
          tc_ld16(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)((2 * i + d) * NMMA + 16 * h), v);
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            const int col = 16 * h + jj;
            acc[col / kNC] += __uint_as_float(v[jj]) *
                              pow2f(FMT == kFmtF8 ? -4 * (col % kNC) : 4 - 2 * (col % kNC));
          }
        }
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars.d_empty[d]);
    const int gi = group_of(a, T32);
    const F4Group gp = group_at(a, gi);
    float out_scale = osc[0];
#pragma unroll
    for (int g = 1; g < kMaxGroups; ++g)
      if (gi == g) out_scale = osc[g];
    const int64_t row = (T - gp.tile0) * kTileRows + row_in_tile;  // row of the group's W and y
    // to true units: (acc * s_w) * 2^-sh (the power of two last: exact
    // unless the result itself under- or overflows)
#pragma unroll
    for (int m = 0; m < MR; ++m) acc[m] = ldexpf(acc[m] * out_scale, -sh[m]);
    if (c0 == 0 && c1 == sk.nch) {  // whole tile in this CTA
      if (row < gp.N) {
#pragma unroll
        for (int m = 0; m < MR; ++m)
          if (m < a.M) gp.y[m * gp.ldy + row] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[m]));
      }
      continue;
    }
    if (a.sched == kSchedCluster) {
      // Part r of the tile's chunks.  Ranks 1..S-1 store their row's partial
      // sums into rank 0's buffer red[r - 1][row] and arrive (one per warp)
      // on its barrier; rank 0 adds them to its own in rank (= K) order.
      const uint32_t rank = cluster_ctarank();
      if (rank != 0) {
        const uint32_t dst =
            cluster_map(smem_u32(red + ((size_t)(rank - 1) * kTileRows + row_in_tile) * MR), 0);
#pragma unroll
        for (int m = 0; m < MR; ++m) st_cluster_f32(dst + 4u * m, acc[m]);
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(cluster_map(smem_u32(&bars.cl_full), 0));
      } else if (__all_sync(0xFFFFFFFFu, mbar_wait_cluster_bounded(&bars.cl_full, 0u, a.status)) &&
                 row < gp.N) {
        for (int r = 1; r < a.ksplit; ++r) {
#pragma unroll
          for (int m = 0; m < MR; ++m) acc[m] += red[((size_t)(r - 1) * kTileRows + row_in_tile) * MR + m];
        }
#pragma unroll
        for (int m = 0; m < MR; ++m)
          if (m < a.M) gp.y[m * gp.ldy + row] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[m]));
      }
      continue;
    }
    // Split tile.  CTAs c_first..c_last share it; each keeps the partial sums
    // of its first and last segment (slots 0 and 1; a single segment uses 0).
    const int c_first = sk.owner(T * sk.nch), c_last = sk.owner(T * sk.nch + sk.nch - 1);
    const int nslot = c_last - c_first + 1;
    // a row's MR partial sums are contiguous: one or a few vector accesses
    auto part_at = [&](int c, int sl) {
      return a.part + ((size_t)(2 * c + sl) * kTileRows + row_in_tile) * MR;
    };
    {
      float *p = part_at(blockIdx.x, j == 0 ? 0 : 1);
      if constexpr (MR == 2) {
        *reinterpret_cast<float2 *>(p) = make_float2(acc[0], acc[1]);
      } else {
#pragma unroll
        for (int m = 0; m < MR; m += 4)
          *reinterpret_cast<float4 *>(p + m) = make_float4(acc[m], acc[m + 1], acc[m + 2], acc[m + 3]);
      }
    }
    // The warps report in (a CTA-scope release); one thread makes the CTA's
    // stores visible device-wide (a cumulative fence) and counts the
    // segment; the tile's last CTA adds the partials in K order.
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars.part_done);
    const uint32_t par = (uint32_t)(n_split & 1);
    ++n_split;
    if (warp == kEpiWarp0 && lane == 0) {
      const bool got = mbar_wait_bounded(&bars.part_done, par, a.status);
      __threadfence();
      *last_flag = got && (a.cnt32 ? atomicAdd(a.cnt32 + T, 1u) == (unsigned)(nslot - 1)
                                    : count_split_segment(a.cnt + T, a.epoch, nslot));
      __threadfence();
      mbar_arrive(&bars.flag_ready);
    }
    if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(&bars.flag_ready, par, a.status))) return false;
    if (*last_flag) {
      __threadfence();
      if (row < gp.N) {
        // Sums in K order, per row of X.  The partials sit in other SMs' L2
        // lines (often across the die boundary), so the loads of several
        // CTAs are put in flight together before any is added.
        auto load_part = [&](int c, float (&v)[MR]) {
          // the tile is the last segment of c_first (its first too if c_first
          // has only one) and the first segment of every later CTA
          int sl = 0;
          if (c == c_first) {
            const int64_t gb = sk.total * c / sk.G, ge = sk.total * (c + 1) / sk.G;
            sl = ((ge - 1) / sk.nch != gb / sk.nch) ? 1 : 0;
          }
          if (c == (int)blockIdx.x && sl == (j == 0 ? 0 : 1)) {
#pragma unroll
            for (int m = 0; m < MR; ++m) v[m] = acc[m];
          } else if constexpr (MR == 2) {
            const float2 q = __ldcg(reinterpret_cast<const float2 *>(part_at(c, sl)));
            v[0] = q.x;
            v[1] = q.y;
          } else {
#pragma unroll
            for (int m = 0; m < MR; m += 4) {
              const float4 q = __ldcg(reinterpret_cast<const float4 *>(part_at(c, sl) + m));
              v[m] = q.x;
              v[m + 1] = q.y;
              v[m + 2] = q.z;
              v[m + 3] = q.w;
            }
          }
        };
        constexpr int GP = MR >= 16 ? 2 : MR >= 8 ? 4 : 8;  // CTAs loaded together
        float t[MR];
#pragma unroll
        for (int m = 0; m < MR; ++m) t[m] = 0.0f;
        for (int c0 = c_first; c0 <= c_last; c0 += GP) {
          float v[GP][MR];
#pragma unroll
          for (int g = 0; g < GP; ++g)
            if (c0 + g <= c_last) load_part(c0 + g, v[g]);
#pragma unroll
          for (int g = 0; g < GP; ++g)
            if (c0 + g <= c_last) {
#pragma unroll
              for (int m = 0; m < MR; ++m) t[m] += v[g][m];
            }
        }
#pragma unroll
        for (int m = 0; m < MR; ++m)
          if (m < a.M) gp.y[m * gp.ldy + row] = __bfloat16_as_ushort(__float2bfloat16_rn(t[m]));
      }
    }
  }
  return true;
}

__device__ __forceinline__ void init_common(F4Bars &bars, int ns, int ni) {
  for (int s = 0; s < ns; ++s) {
    mbar_init(&bars.full[s], 1);
    mbar_init(&bars.empty[s], 1);
    mbar_init(&bars.sf_ready[s], 1);
  }
  for (int i = 0; i < ni; ++i) {
    mbar_init(&bars.d_full[i][0], 1);
    mbar_init(&bars.d_full[i][1], 1);
    mbar_init(&bars.drain[i], 1);
  }
  mbar_init(&bars.d_empty[0], 4);
  mbar_init(&bars.d_empty[1], 4);
  mbar_init(&bars.part_done, 4);
  mbar_init(&bars.flag_ready, 1);
  fence_mbar_init();
}

// ---- streamed-B path -----------------------------------------------------------

// X -> NVFP4 components in the workspace.  Grid (blocks of K / 256 threads,
// M); every CTA finds its row's max|x|, then each thread splits one block.
__global__ void __launch_bounds__(kXsplitThreads)
    xsplit_kernel(const uint16_t *x, int64_t ldx, int M, int64_t K, int nmma, uint8_t *bcodes,
                  uint8_t *sfb, int32_t *sh_out, const uint16_t *x2, int64_t ldx2) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // X may come from the previous kernel, and the previous GEMV may still
  // read the workspace: wait for it before touching either.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __shared__ uint32_t red[kXsplitThreads / 32];
  const int m = blockIdx.y;
  const uint16_t *xr = x + m * ldx;
  // x2 (optional): X is silu(x) * x2, computed where it is read
  const uint16_t *ur = x2 ? x2 + m * ldx2 : nullptr;
  auto ld8 = [&](int64_t i) {
    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(xr) + i);
    return ur ? swiglu_bf16x8(v, __ldg(reinterpret_cast<const uint4 *>(ur) + i)) : v;
  };
  const int64_t nb = K / 16;
  uint32_t mx = 0;
  for (int64_t i = threadIdx.x; i < K / 8; i += kXsplitThreads) mx = max(mx, absmax_bf16x8(ld8(i)));
  for (int o = 16; o; o >>= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
  __syncthreads();
  mx = 0;
  for (int w = 0; w < kXsplitThreads / 32; ++w) mx = max(mx, red[w]);
  const int sh = prescale_exponent(mx);
  if (blockIdx.x == 0 && threadIdx.x == 0) sh_out[m] = sh;

  const int64_t b = (int64_t)blockIdx.x * kXsplitThreads + threadIdx.x;
  const int64_t KH = K / 2;
  if (b < nb) {
    uint2 code[kNC];
    uint32_t sb[kNC];
    const uint4 v[2] = {ld8(2 * b), ld8(2 * b + 1)};
    split_block_regs(v, sh, code, sb);
    // atom position of this block: K64 step b / 4, block b % 4
    uint8_t *atom = sfb + (b >> 2) * 512 + (b & 3);
#pragma unroll
    for (int c = 0; c < kNC; ++c) {
      const int n = m * kNC + c;
      *reinterpret_cast<uint2 *>(bcodes + n * KH + 8 * b) = code[c];
      atom[16 * (n & 31) + 4 * ((n >> 5) & 3)] = (uint8_t)sb[c];
    }
  }
  // operand rows past the last component: zero scales (their codes then
  // contribute nothing)
  if (m == M - 1 && blockIdx.x == 0)
    for (int64_t i = threadIdx.x; i < (K / 64) * (nmma - M * kNC); i += kXsplitThreads) {
      const int64_t t = i / (nmma - M * kNC);
      const int n = M * kNC + (int)(i % (nmma - M * kNC));
      *reinterpret_cast<uint32_t *>(sfb + t * 512 + 16 * (n & 31) + 4 * ((n >> 5) & 3)) = 0u;
    }
}

template <int NMMA, bool PREP>
__global__ void __launch_bounds__(kThreads, 1)
    gemv_f4_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_ws,
                   const __grid_constant__ CUtensorMap tm_b, const F4Args a) {
  using L = StageS<NMMA>;
  constexpr int NI = CfgS<NMMA>::NI, NS = CfgS<NMMA>::NS;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment for the swizzled tiles
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  F4Bars &bars = *reinterpret_cast<F4Bars *>(smem + NS * L::BYTES);
  // kSchedCluster: the other ranks' partial sums, [rank - 1][128 rows][N_MMA / 8]
  float *red = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(&bars) +
                                         ((sizeof(F4Bars) + 15) & ~size_t(15)));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const StreamK sk(a.n_tiles, a.n_chunks, a.sched, a.ksplit);

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) {
    mbar_init(&bars.cl_full, a.sched == kSchedCluster ? 4 * (a.ksplit - 1) : 1);
    init_common(bars, NS, NI);
  }
  if (warp == 0) tmem_alloc(&bars.tmem);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem;
  // the cluster's barriers are initialized before any rank arrives remotely
  if (a.sched == kSchedCluster) cluster_sync_all();

  if (warp == kProducerS) {
    if (lane == 0) {
      if (!PREP) {
        prefetch_tmap(&tm_w);
        prefetch_tmap(&tm_ws);
      }
      prefetch_tmap(&tm_b);
      // processing position i -> ring slot i % NS, stage stage_of(i)
      PreparedTile src, psrc;
      auto load_w = [&](int i) {
        const int s = i % NS;
        uint8_t *stg = smem + (size_t)s * L::BYTES;
        int tile, ch;
        sk.tile_ch(sk.stage_of(i), tile, ch);
        const int row0 = tile * kTileRows;
        mbar_arrive_expect_tx(&bars.full[s], L::TX);
        if (PREP) {
          src.at(a, tile, sk.nch);
          bulk_g2s(stg + L::W, src.wc + (size_t)ch * 16384, 16384u, &bars.full[s]);
          bulk_g2s(stg + L::SFA, src.wsa + (size_t)ch * 2048, 2048u, &bars.full[s]);
        } else {
          tma_load_2d(stg + L::W, &tm_w, ch * (kChunkK / 2), row0, &bars.full[s]);
          tma_load_2d(stg + L::RAW, &tm_ws, ch * (kChunkK / 16), row0, &bars.full[s]);
        }
      };
      auto load_x = [&](int i) {
        const int s = i % NS;
        uint8_t *stg = smem + (size_t)s * L::BYTES;
        int tile, ch;
        sk.tile_ch(sk.stage_of(i), tile, ch);
        tma_load_2d(stg + L::B, &tm_b, ch * (kChunkK / 2), 0, &bars.full[s]);
        bulk_g2s(stg + L::SFB, a.sfb + (size_t)ch * 2048, 2048u, &bars.full[s]);
      };
      auto prefetch_w = [&](int i) {
        int tile, ch;
        sk.tile_ch(sk.stage_of(i), tile, ch);
        if (PREP) {
          psrc.at(a, tile, sk.nch);
          bulk_prefetch_l2(psrc.wc + (size_t)ch * 16384, 16384u);
          bulk_prefetch_l2(psrc.wsa + (size_t)ch * 2048, 2048u);
        } else {
          tma_prefetch_l2_2d(&tm_w, ch * (kChunkK / 2), tile * kTileRows);
          tma_prefetch_l2_2d(&tm_ws, ch * (kChunkK / 16), tile * kTileRows);
        }
      };
      // W of the first stages before the previous kernel has finished, and
      // more W into L2: HBM keeps streaming while X is being split.
      const int pre = min(NS, sk.n_st);
      for (int i = 0; i < pre; ++i) load_w(i);
      for (int i = pre; i < min(pre + kPrefetch, sk.n_st); ++i) prefetch_w(i);
      asm volatile("griddepcontrol.wait;" ::: "memory");
      for (int i = 0; i < pre; ++i) load_x(i);
      int i = pre;
      for (; i < sk.n_st; ++i) {
        const int s = i % NS;
        if (!mbar_wait_bounded(&bars.empty[s], (uint32_t)((i / NS - 1) & 1), a.status)) break;
        load_w(i);
        load_x(i);
      }
      // never leave with copies in flight
      for (int k = (i > NS ? i - NS : 0); k < i; ++k)
        mbar_wait_bounded(&bars.full[k % NS], (uint32_t)((k / NS) & 1), a.status);
    }
  } else if (warp < NI) {
    const uint32_t sbase = smem_u32(smem);
    const uint64_t dB0 = sdesc(sbase + L::B, 16, 1024, kSw128);
    const uint64_t dSB0 = sdesc(sbase + L::SFB, 0, 128, kNoSwizzle);
    auto b_desc = [&](int i, int, int t) {
      return dB0 + (uint64_t)((i % NS) * (L::BYTES >> 4)) + 2u * t;
    };
    auto sfb_desc = [&](int i, int, int t) {
      return dSB0 + (uint64_t)((i % NS) * (L::BYTES >> 4)) + 32u * t;
    };
    issuer_loop<NI, NS, NMMA, PREP, L>(smem, bars, tmem, sk, warp, lane, a.status, b_desc,
                                          sfb_desc, [](int) { return true; });
  } else if (warp == kRelayWarp) {
    if (!PREP) relay_loop<NS, L>(smem, bars, sk, lane, a.status);
  } else if (warp >= kEpiWarp0) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    int sh[kMaxRowsX] = {};
#pragma unroll
    for (int m = 0; m < NMMA / kNC; ++m)
      if (m < a.M) sh[m] = a.sh[m];
    int n_split = 0;
    epilogue_loop<NI, NMMA>(a, bars, tmem, sk, warp, lane, sh, red, 0, 0, n_split);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_free(tmem);
  }
  // no rank leaves while another may still write into its shared memory
  if (a.sched == kSchedCluster) cluster_sync_all();
}

// ---- resident-B path (M <= 2) ---------------------------------------------------

// One 256-element chunk of row m of X -> its eight NVFP4 components in a B
// slot image (codes: 16 operand rows x 128 B, row n at 128 n with its
// 16-byte unit u at u ^ (n % 8); scales: four K64 steps of 16 lines of 16 B),
// in shared or global memory.  One warp: lane 2 b + h holds elements
// 8 h .. 8 h + 7 of the chunk's block b (v).  The last row of X also zeroes
// the operand rows after its components.
__device__ __forceinline__ void split_chunk_slot(const uint4 v, int sh, int m, int M, uint8_t *codes,
                                                 uint8_t *sf, int lane) {
  const int bb = lane >> 1, hf = lane & 1;
  const float p1 = pow2f(sh / 2), p2 = pow2f(sh - sh / 2);
  float r[8];
  {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      r[2 * t] = bf16_bits_to_f32(w[t] & 0xFFFFu) * p1 * p2;
      r[2 * t + 1] = bf16_bits_to_f32(w[t] >> 16) * p1 * p2;
    }
  }
#pragma unroll
  for (int c = 0; c < kNC; ++c) {
    const int n = m * kNC + c;
    float m4[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) m4[e] = fmaxf(fabsf(r[e]), fabsf(r[e + 4]));
    float amax = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));  // the block's other half
    // Any scale is valid -- the residual tracks what was taken -- so an
    // approximate reciprocal stands in for the division.
    const uint32_t sb = f32_to_e4m3_satfinite(amax * (1.0f / 6.0f) * pow2f(2 * c - 4));
    const float d = e4m3_to_f32(sb) * pow2f(4 - 2 * c);
    uint32_t cw = 0u;
    if (d > 0.0f) {
      float inv;
      asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(inv) : "f"(d));
      float q[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) q[e] = r[e] * inv;
      cw = f32x8_to_e2m1_packed(q);
      uint32_t e2[4];
      e2m1x8_to_f16x2x4(cw, e2);
#pragma unroll
      for (int t = 0; t < 4; ++t) {  // e2m1 * d is exact; one rounding per update
        r[2 * t] = fmaf(-f16lo_to_f32(e2[t]), d, r[2 * t]);
        r[2 * t + 1] = fmaf(-f16hi_to_f32(e2[t]), d, r[2 * t + 1]);
      }
    }
    *reinterpret_cast<uint32_t *>(codes + n * 128 + (((bb >> 1) ^ (n & 7)) << 4) + 8 * (bb & 1) +
                                  4 * hf) = cw;
    // the four scales of K64 step t sit in lanes 8 t, 8 t + 2, 8 t + 4, 8 t + 6
    const uint32_t s1 = __shfl_down_sync(0xFFFFFFFFu, sb, 2);
    const uint32_t s2 = __shfl_down_sync(0xFFFFFFFFu, sb, 4);
    const uint32_t s3 = __shfl_down_sync(0xFFFFFFFFu, sb, 6);
    if ((lane & 7) == 0)
      *reinterpret_cast<uint4 *>(sf + (lane >> 3) * 256 + 16 * n) =
          make_uint4(sb | s1 << 8 | s2 << 16 | s3 << 24, 0u, 0u, 0u);
  }
  if (m == M - 1 && M * kNC < 16) {
    // operand rows after the last component: zero codes and scale lines
    const int n0 = M * kNC, nr = 16 - n0;
    uint4 *zc = reinterpret_cast<uint4 *>(codes + n0 * 128);
    for (int i = lane; i < nr * 8; i += 32) zc[i] = make_uint4(0, 0, 0, 0);
    for (int i = lane; i < 4 * nr; i += 32)
      *reinterpret_cast<uint4 *>(sf + (i / nr) * 256 + 16 * (n0 + i % nr)) = make_uint4(0, 0, 0, 0);
  }
}


// X (M <= 2 rows) -> B slot images of every K chunk, once per call.  Grid
// (chunks / kSplitWarps rounded up, M); CTA (j, m) finds row m's max|x| (the
// prescale 2^sh puts it in [2^14, 2^15)), then warp w splits chunk
// kSplitWarps j + w of row m into its eight components: lane 2 b + h holds
// elements 8 h .. 8 h + 7 of the chunk's block b.  Writes the images' rows
// 8 m .. 8 m + 7 (and, for the last row of X, zeros in the rows after it) and
// sh[m].
__global__ void __launch_bounds__(128 * kSplitWarps)
    xsplit_slots_kernel(const uint16_t *x, int64_t ldx, int M, int64_t K, uint8_t *slot_codes,
                        uint8_t *slot_sf, int32_t *sh_out, int32_t *status, const uint16_t *x2,
                        int64_t ldx2) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  extern __shared__ uint4 xrow[];  // row m of X (K bf16), staged once
  __shared__ uint64_t bar;
  __shared__ uint32_t red[32];
  const int m = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nt = blockDim.x;  // 32 kSplitWarps, or 4x that to form silu(x) * x2 sooner
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  // X may come from the previous kernel, and the previous GEMV may still
  // read the workspace: wait for it before touching either.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // The row in one bulk copy: a single memory round trip, which matters
  // because the next GEMV's weight stream is already filling the memory
  // queues when this kernel runs.  With x2, X = silu(x) * x2: both rows
  // staged, then combined in place by all the CTA's threads (every CTA
  // forms the whole row: its max sets the prescale).
  uint4 *urow = xrow + K / 8;
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(&bar, (uint32_t)(K * 2) * (x2 ? 2u : 1u));
    bulk_g2s(xrow, x + m * ldx, (uint32_t)(K * 2), &bar);
    if (x2) bulk_g2s(urow, x2 + m * ldx2, (uint32_t)(K * 2), &bar);
  }
  if (!mbar_wait_bounded(&bar, 0u, status)) return;
  if (x2) {
    for (int i = threadIdx.x; i < (int)(K / 8); i += nt) xrow[i] = swiglu_bf16x8(xrow[i], urow[i]);
    __syncthreads();
  }
  uint32_t mx = 0;
  for (int i = threadIdx.x; i < (int)(K / 8); i += nt) mx = max(mx, absmax_bf16x8(xrow[i]));
  for (int o = 16; o; o >>= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
  if (lane == 0) red[warp] = mx;
  __syncthreads();
  mx = 0;
  for (int w = 0; w < nt / 32; ++w) mx = max(mx, red[w]);
  const int sh = prescale_exponent(mx);
  if (blockIdx.x == 0 && threadIdx.x == 0) sh_out[m] = sh;

  const int ch = blockIdx.x * kSplitWarps + warp;
  if (warp >= kSplitWarps || ch >= (int)(K / kChunkK)) return;
  const int bb = lane >> 1, hf = lane & 1;
  split_chunk_slot(xrow[(ch * kChunkK + 16 * bb + 8 * hf) / 8], sh, m, M,
                   slot_codes + (size_t)ch * 2048, slot_sf + (size_t)ch * 1024, lane);
}

// Two signed floats -> two E4M3 bytes (element 0 in the low byte), round to
// nearest even, saturating.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2_rn(float lo, float hi) {
  uint32_t out;
  asm("{\n.reg .b16 r;\ncvt.rn.satfinite.e4m3x2.f32 r, %2, %1;\ncvt.u32.u16 %0, r;\n}"
      : "=r"(out)
      : "f"(lo), "f"(hi));
  return out;
}

// X (M <= 2 rows) -> B slot images for an FP8 weight, once per call:
//   x * 2^sh = sum_{c < 8} 2^(-4c) * e4m3(q_c),
// component c the E4M3 rounding (nearest even) of 2^(4c) times what
// components 0..c-1 left, the residual updated with the exact product; the
// prescale 2^sh puts the row's max|x| in [2^7, 2^8), below the E4M3 maximum.
// A slot holds one 128-element chunk: 16 operand rows x 128 B, row 8 m + c
// = component c of row m, element e at byte e of its row with the 16-byte
// unit u stored at u ^ (n % 8).  Grid (chunks / kSplitWarps rounded up, M);
// warp w splits chunk kSplitWarps j + w, lane l elements 4 l .. 4 l + 3.
__global__ void __launch_bounds__(32 * kSplitWarps)
    xsplit_f8_kernel(const uint16_t *x, int64_t ldx, int M, int64_t K, uint8_t *slot_codes,
                     int32_t *sh_out, int32_t *status) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  extern __shared__ uint4 xrow[];  // row m of X (K bf16), staged once
  __shared__ uint64_t bar;
  __shared__ uint32_t red[kSplitWarps];
  const int m = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  // X may come from the previous kernel, and the previous GEMV may still
  // read the workspace: wait for it before touching either.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(&bar, (uint32_t)(K * 2));
    bulk_g2s(xrow, x + m * ldx, (uint32_t)(K * 2), &bar);
  }
  if (!mbar_wait_bounded(&bar, 0u, status)) return;
  uint32_t mx = 0;
  for (int i = threadIdx.x; i < (int)(K / 8); i += 32 * kSplitWarps) mx = max(mx, absmax_bf16x8(xrow[i]));
  for (int o = 16; o; o >>= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
  if (lane == 0) red[warp] = mx;
  __syncthreads();
  mx = 0;
  for (int w = 0; w < kSplitWarps; ++w) mx = max(mx, red[w]);
  const int sh = mx ? prescale_exponent(mx) - 7 : 0;  // max in [2^7, 2^8)
  if (blockIdx.x == 0 && threadIdx.x == 0) sh_out[m] = sh;

  const int ch = blockIdx.x * kSplitWarps + warp;
  if (ch >= (int)(K / 128)) return;
  const uint2 v = reinterpret_cast<const uint2 *>(xrow)[ch * 32 + lane];
  const float p1 = pow2f(sh / 2), p2 = pow2f(sh - sh / 2);
  float r[4] = {bf16_bits_to_f32(v.x & 0xFFFFu) * p1 * p2, bf16_bits_to_f32(v.x >> 16) * p1 * p2,
                bf16_bits_to_f32(v.y & 0xFFFFu) * p1 * p2, bf16_bits_to_f32(v.y >> 16) * p1 * p2};
  uint8_t *codes = slot_codes + (size_t)ch * 2048;
#pragma unroll
  for (int c = 0; c < kNC; ++c) {
    const int n = m * kNC + c;
    const float up = pow2f(4 * c), down = pow2f(-4 * c);
    const uint32_t lo = f32x2_to_e4m3x2_rn(r[0] * up, r[1] * up);
    const uint32_t hi = f32x2_to_e4m3x2_rn(r[2] * up, r[3] * up);
    const uint32_t hl = e4m3x2_to_f16x2(lo), hh = e4m3x2_to_f16x2(hi);
    r[0] = fmaf(-f16lo_to_f32(hl), down, r[0]);  // e4m3 * 2^-4c is exact; one rounding
    r[1] = fmaf(-f16hi_to_f32(hl), down, r[1]);
    r[2] = fmaf(-f16lo_to_f32(hh), down, r[2]);
    r[3] = fmaf(-f16hi_to_f32(hh), down, r[3]);
    *reinterpret_cast<uint32_t *>(codes + n * 128 + (((lane >> 2) ^ (n & 7)) << 4) + 4 * (lane & 3)) =
        lo | hi << 16;
  }
  if (m == M - 1 && M * kNC < 16) {
    // operand rows after the last component: zero
    const int n0 = M * kNC, nr = 16 - n0;
    uint4 *zc = reinterpret_cast<uint4 *>(codes + n0 * 128);
    for (int i = lane; i < nr * 8; i += 32) zc[i] = make_uint4(0, 0, 0, 0);
  }
}

template <bool PREP, int FMT = kFmtNv, bool SPLIT = false>
__global__ void __launch_bounds__(kThreads, 1)
    gemv_f4r_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_ws,
                    const F4Args a) {
  using L = StageRT<FMT>;
  constexpr uint32_t kSlotSf = FmtR<FMT>::kSlotSf;
  static_assert(FMT == kFmtNv || !PREP, "FP8 weights are read row-major");
  constexpr int NMMA = 16;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t *bcodes = smem + kNSR * L::BYTES;                   // [slot][16 rows][128 B], swizzled
  uint8_t *bsf = bcodes + (size_t)a.n_slots * 2048;           // NVFP4: [slot][4 steps][256 B] + pad
  F4Bars &bars = *reinterpret_cast<F4Bars *>(bsf + (size_t)a.n_slots * kSlotSf + 256);
  // kSchedCluster: the other ranks' partial sums, [rank - 1][128 rows][2]
  float *red = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(&bars) +
                                         ((sizeof(F4Bars) + 15) & ~size_t(15)));
  F4SplitBars &sbars = *reinterpret_cast<F4SplitBars *>(
      red + (a.sched == kSchedCluster ? (size_t)(a.ksplit - 1) * kTileRows * 2 : 0));
  static_assert(!SPLIT || FMT == kFmtNv, "the kernel splits NVFP4 components only");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const StreamK sk(a.n_tiles, a.n_chunks, a.sched, a.ksplit);
  // B slot of chunk ch: this CTA's chunks run consecutively from ch_begin
  const int ch_begin = sk.ch0;
  auto slot_of = [&](int st) { return st % sk.nch; };

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) {
    mbar_init(&bars.b_ready, 1);
    mbar_init(&bars.cl_full, a.sched == kSchedCluster ? 4 * (a.ksplit - 1) : 1);
    if (SPLIT)
      for (int j = 0; j < a.n_slots; ++j) mbar_init(&sbars.slot_ready[j], 1);
    init_common(bars, kNSR, kIssuersR);
  }
  if (warp == 0) tmem_alloc(&bars.tmem);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem;
  // the cluster's barriers are initialized before any rank arrives remotely
  if (a.sched == kSchedCluster) cluster_sync_all();

  if (warp == kProducerR) {
    // W only: it is never written on the stream, so no wait for the
    // previous kernel.
    if (lane == 0) {
      if (!PREP) {
        prefetch_tmap(&tm_w);
        if (FMT == kFmtNv) prefetch_tmap(&tm_ws);
      }
      // processing position i -> ring slot i % NS, stage stage_of(i).  The
      // source of a stage is worked out before its slot frees (where), so
      // the copies go out the moment it does (issue): the slot's turnaround
      // bounds the bytes in flight.
      PreparedTile src;
      struct Src {
        const uint8_t *w, *sf;  // prepared weight
        int ch, row0;           // row-major weight (tensor-map coordinates)
      };
      auto where = [&](int i) {
        Src r;
        int tile;
        sk.tile_ch(sk.stage_of(i), tile, r.ch);
        r.row0 = tile * kTileRows;
        if (PREP) {
          src.at(a, tile, sk.nch);
          r.w = src.wc + (size_t)r.ch * 16384;
          r.sf = src.wsa + (size_t)r.ch * 2048;
        }
        return r;
      };
      auto issue = [&](int i, const Src &r) {
        const int s = i % kNSR;
        uint8_t *stg = smem + (size_t)s * L::BYTES;
        mbar_arrive_expect_tx(&bars.full[s], L::TX);
        if (PREP) {
          bulk_g2s(stg + L::W, r.w, 16384u, &bars.full[s]);
          bulk_g2s(stg + L::SFA, r.sf, 2048u, &bars.full[s]);
        } else {
          // 128 bytes of each row per stage: 256 NVFP4 or 128 FP8 elements
          tma_load_2d(stg + L::W, &tm_w, r.ch * 128, r.row0, &bars.full[s]);
          if (FMT == kFmtNv)
            tma_load_2d(stg + L::RAW, &tm_ws, r.ch * (kChunkK / 16), r.row0, &bars.full[s]);
        }
      };
      // The ring alone keeps W in flight: an extra L2 prefetch at the start
      // only lengthened the queues every later access (X, B, the fix-ups)
      // waits in.
      const int pre = min(kNSR, sk.n_st);
      for (int i = 0; i < pre; ++i) issue(i, where(i));
      int i = pre;
      for (; i < sk.n_st; ++i) {
        const int s = i % kNSR;
        const Src r = where(i);
        if (!mbar_wait_bounded(&bars.empty[s], (uint32_t)((i / kNSR - 1) & 1), a.status)) break;
        issue(i, r);
      }
      for (int k = (i > kNSR ? i - kNSR : 0); k < i; ++k)
        mbar_wait_bounded(&bars.full[k % kNSR], (uint32_t)((k / kNSR) & 1), a.status);
    }
  } else if (SPLIT && (warp == kLoaderWarpR || warp == kSplitWarpX || warp >= kEpiWarp0)) {
    // ---- NVFP4 with at most six slots: X split into components here, one
    // slot per warp, while the ring fills (no split launch, no slot copy).
    // Six warps (5, 7 and the epilogue warps, which go on to the epilogue);
    // the prescale comes from this CTA's chunks of each row of X (all ranks
    // and CTAs leave their sums in true units).  With more slots the split
    // kernel's many warps finish them sooner than six warps here would.
    const int widx = warp == kLoaderWarpR ? 0 : warp - kSplitWarpX + 1;
    const int bb = lane >> 1, hf = lane & 1;
    if (widx == 0 && lane < 16)  // read (into lanes no N = 16 MMA uses) after the last slot
      reinterpret_cast<uint4 *>(bsf + (size_t)a.n_slots * kSlotSf)[lane] = make_uint4(0, 0, 0, 0);
    asm volatile("griddepcontrol.wait;" ::: "memory");  // X may come from the previous kernel
    // split warp w: slot w (a.n_slots <= kSplitW)
    const int j = widx;
    uint4 v[2];
    uint32_t mx[2] = {0u, 0u};
    if (j < a.n_slots) {
      const int ch = (ch_begin + j) % sk.nch;
#pragma unroll
      for (int m = 0; m < 2; ++m)
        if (m < a.M) {
          v[m] = __ldcg(reinterpret_cast<const uint4 *>(a.x + m * a.ldx + (int64_t)ch * kChunkK +
                                                       16 * bb + 8 * hf));
          mx[m] = absmax_bf16x8(v[m]);
        }
    }
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      for (int o = 16; o; o >>= 1) mx[m] = max(mx[m], __shfl_xor_sync(0xFFFFFFFFu, mx[m], o));
      if (lane == 0) sbars.xmax[widx][m] = mx[m];
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the pad
    asm volatile("bar.sync 1, %0;" ::"n"(32 * kSplitW) : "memory");
    int sh[kMaxRowsX] = {};
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      uint32_t r = 0;
#pragma unroll
      for (int w = 0; w < kSplitW; ++w) r = max(r, sbars.xmax[w][m]);
      sh[m] = prescale_exponent(r);
    }
    if (j < a.n_slots) {
#pragma unroll
      for (int m = 0; m < 2; ++m)
        if (m < a.M)
          split_chunk_slot(v[m], sh[m], m, a.M, bcodes + (size_t)j * 2048, bsf + (size_t)j * 1024,
                           lane);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // read by tcgen05.mma / .cp
      __syncwarp();
      if (lane == 0) mbar_arrive(&sbars.slot_ready[j]);
    }
    int n_split = 0;
    if (warp >= kEpiWarp0)
      epilogue_loop<kIssuersR, NMMA, FMT>(a, bars, tmem, sk, warp, lane, sh, red, 0, 0, n_split);
  } else if (warp == kLoaderWarpR) {
    // ---- warp 5: the zero pad after the last slot's scales, then (once the
    // split kernel has finished) this CTA's B slots: chunks ch_begin,
    // ch_begin + 1, ... (mod K / 256), contiguous in the workspace up to the
    // wrap-around, so at most two copies per array.
    if (FMT == kFmtNv && lane < 16)
      reinterpret_cast<uint4 *>(bsf + (size_t)a.n_slots * kSlotSf)[lane] = make_uint4(0, 0, 0, 0);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the pad is read by tcgen05.cp
    __syncwarp();
    if (lane == 0) {
      asm volatile("griddepcontrol.wait;" ::: "memory");
      const int n1 = min(a.n_slots, sk.nch - ch_begin), n2 = a.n_slots - n1;
      mbar_arrive_expect_tx(&bars.b_ready, (uint32_t)a.n_slots * (2048u + kSlotSf));
      bulk_g2s(bcodes, a.slot_codes + (size_t)ch_begin * 2048, (uint32_t)n1 * 2048u, &bars.b_ready);
      if (FMT == kFmtNv)
        bulk_g2s(bsf, a.sfb + (size_t)ch_begin * kSlotSf, (uint32_t)n1 * kSlotSf, &bars.b_ready);
      if (n2 > 0) {
        bulk_g2s(bcodes + (size_t)n1 * 2048, a.slot_codes, (uint32_t)n2 * 2048u, &bars.b_ready);
        if (FMT == kFmtNv)
          bulk_g2s(bsf + (size_t)n1 * kSlotSf, a.sfb, (uint32_t)n2 * kSlotSf, &bars.b_ready);
      }
      // never leave with copies in flight
      mbar_wait_bounded(&bars.b_ready, 0u, a.status);
    }
  } else if (warp == kRelayWarp) {
    if (!PREP && FMT == kFmtNv) relay_loop<kNSR, L>(smem, bars, sk, lane, a.status);
  } else if (warp >= kEpiWarp0) {
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the split kernel wrote sh
    int sh[kMaxRowsX] = {};
#pragma unroll
    for (int m = 0; m < 2; ++m)
      if (m < a.M) sh[m] = a.sh[m];
    int n_split = 0;
    epilogue_loop<kIssuersR, NMMA, FMT>(a, bars, tmem, sk, warp, lane, sh, red, 0, 0, n_split);
  } else if (warp < kIssuersR) {
    // ---- MMA issuers: each stage waits for its B slot
    const uint64_t dB0 = sdesc(smem_u32(bcodes), 16, 1024, kSw128);
    const uint64_t dSB0 = sdesc(smem_u32(bsf), 0, 128, kNoSwizzle);
    auto b_desc = [&](int, int st, int t) { return dB0 + (uint64_t)(slot_of(st) * (2048 >> 4)) + 2u * t; };
    auto sfb_desc = [&](int, int st, int t) {
      return dSB0 + (uint64_t)(slot_of(st) * (1024 >> 4)) + (uint64_t)(16u * t);
    };
    // one barrier for all slots (copied in), or one per slot (split here)
    auto b_wait = [&](int st) {
      return SPLIT ? mbar_wait_bounded(&sbars.slot_ready[slot_of(st)], 0u, a.status)
                   : mbar_wait_bounded(&bars.b_ready, 0u, a.status);
    };
    if constexpr (FMT == kFmtNv)
      issuer_loop<kIssuersR, kNSR, NMMA, PREP, L>(smem, bars, tmem, sk, warp, lane, a.status,
                                                  b_desc, sfb_desc, b_wait);
    else
      issuer_loop_f8<kIssuersR, kNSR, NMMA, L>(smem, bars, tmem, sk, warp, lane, a.status, b_desc,
                                               b_wait);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_free(tmem);
  }
  // no rank leaves while another may still write into its shared memory
  if (a.sched == kSchedCluster) cluster_sync_all();
}

// ---- chained decode calls (one persistent launch) --------------------------------
//
// A decode step is a chain of GEMVs in which a call's X may be the previous
// call's output (a layer's gate projection feeding its down projection, the
// last layer feeding the LM head).  Launched one by one, every call pays a
// kernel boundary: its CTAs start only when the previous call's leave the
// SMs and the first weight bytes land microseconds later.  Here one launch
// of one CTA per SM runs the calls in turn: the producer streams the next
// call's weight into the ring as slots free (a weight is never written on
// the stream, so it needs no wait), and only the MMAs of a call whose X is
// the previous call's output wait, for a per-call count of finished CTAs in
// the workspace.  Every CTA splits the K chunks of X it needs itself (seven
// warps, in rounds; the issuers take each slot as soon as its round wrote
// it), with its own prescale, so its partial sums leave in true units; a
// call with the same X and chunks as the previous one keeps its slots.  The
// B slots fill the shared memory the 8-stage ring leaves, so a call's split
// waits until this CTA's MMAs of the previous call completed: the split and
// its load of X sit between the calls (~3 us), as the separate split kernel
// does between separate calls.  Split tiles of stream-K calls are counted
// with plain atomic adds on counters the launch's first CTA clears (a
// compare-and-swap counter under four contenders cost microseconds).
// The CTAs wait for each other, so all of them must be resident at once:
// one per SM (shared memory allows no second) and grid = SM count.  A
// cooperative launch would guarantee it but measured ~3.5 us slower per
// launch (it gives up the overlap with the previous kernel); the waits are
// bounded instead.
constexpr int kMaxChain = 4;
constexpr int kChainSplitW = 7;  // warps 5, 6, 7 and 8..11 split X
constexpr int kChainSlots = FmtR<kFmtNv>::kMaxSlots;
// The chain's counters (workspace).  CTA 0 clears them at the start of a
// launch and then publishes the launch's epoch in `ready`; every CTA waits
// for that before it counts or reads a count, so a count left by another
// launch, or whatever the workspace held, is never taken for this one's.
// The last CTA to finish sets `ready` back to 0 (a graph replay reuses the
// epoch).  Plain atomic adds: no compare-and-swap retries under contention.
struct ChainCounters {
  unsigned long long ready;
  unsigned int done[kMaxChain];  // CTAs done with call c
  unsigned int finished;         // CTAs past their last wait
};
struct F4Chain {
  F4Args call[kMaxChain];
  int n_calls;
  int dep[kMaxChain];          // 1: call c reads call c - 1's output (wait for it)
  int reuse[kMaxChain];        // 1: call c reads the same X and K chunks as call c - 1
  int n_slots;                 // B slot images in shared memory (the most any call needs)
  ChainCounters *cnt;          // in the workspace
  unsigned long long epoch;    // unique per launch
};
struct F4ChainBars {
  uint64_t slot_ready[kChainSlots];  // one phase per split (none for a call that keeps the slots)
  uint32_t xmax[kChainSplitW][2];
};

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long *p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned int ld_acquire_u32(const unsigned int *p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Bounded wait until *p >= want (acquire); v: the value of an 8-byte word
// (ready) or of a 4-byte count.
__device__ __forceinline__ bool chain_wait_ready(const ChainCounters *k, unsigned long long epoch,
                                                 int32_t *status) {
  if (ld_acquire_u64(&k->ready) == epoch) return true;
  const uint64_t t0 = globaltimer_ns();
  while (ld_acquire_u64(&k->ready) != epoch) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      report(status, IMP_DEV_TIMEOUT);
      return false;
    }
    __nanosleep(64);
  }
  return true;
}
__device__ __forceinline__ bool chain_wait_count(const unsigned int *c, unsigned int want,
                                                 int32_t *status) {
  if (ld_acquire_u32(c) >= want) return true;
  const uint64_t t0 = globaltimer_ns();
  while (ld_acquire_u32(c) < want) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      report(status, IMP_DEV_TIMEOUT);
      return false;
    }
    __nanosleep(64);
  }
  return true;
}

// The split warps' share of one call: this CTA's B slots j < a.n_slots
// (slot j = K chunk (ch0 + j) mod nch, as the issuers read them), warp w
// taking slots w, w + 7, ...; the prescale of row m from this CTA's chunks.
// Every slot barrier j < n_all gets one arrival per call.
__device__ __forceinline__ void chain_split(const F4Args &a, int ch0, int nch, int n_all, int w,
                                            int lane, F4ChainBars &cb, uint8_t *bcodes,
                                            uint8_t *bsf, int (&sh)[kMaxRowsX]) {
  constexpr int R = (kChainSlots + kChainSplitW - 1) / kChainSplitW;
  const int bb = lane >> 1, hf = lane & 1;
  uint4 v[R][2];
  uint32_t mx[2] = {0u, 0u};
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int j = w + kChainSplitW * r;
    if (j < a.n_slots) {
      const int chn = (ch0 + j) % nch;
#pragma unroll
      for (int m = 0; m < 2; ++m)
        if (m < a.M) {
          // L2 only: X may have been written by other SMs in this launch
          const int64_t e = (int64_t)chn * kChunkK + 16 * bb + 8 * hf;
          v[r][m] = __ldcg(reinterpret_cast<const uint4 *>(a.x + m * a.ldx + e));
          if (a.x2)  // X = silu(x) * x2 (a down projection after gate and up)
            v[r][m] = swiglu_bf16x8(v[r][m],
                                    __ldcg(reinterpret_cast<const uint4 *>(a.x2 + m * a.ldx2 + e)));
          mx[m] = max(mx[m], absmax_bf16x8(v[r][m]));
        }
    }
  }
#pragma unroll
  for (int m = 0; m < 2; ++m) {
    for (int o = 16; o; o >>= 1) mx[m] = max(mx[m], __shfl_xor_sync(0xFFFFFFFFu, mx[m], o));
    if (lane == 0) cb.xmax[w][m] = mx[m];
  }
  asm volatile("bar.sync 1, %0;" ::"n"(32 * kChainSplitW) : "memory");
#pragma unroll
  for (int m = 0; m < 2; ++m) {
    uint32_t r = 0;
#pragma unroll
    for (int i = 0; i < kChainSplitW; ++i) r = max(r, cb.xmax[i][m]);
    sh[m] = prescale_exponent(r);
  }
  // round r makes slots 7 r .. 7 r + 6 ready: the issuers, which take the
  // slots in order, start after the first round
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int j = w + kChainSplitW * r;
    if (j < a.n_slots) {
#pragma unroll
      for (int m = 0; m < 2; ++m)
        if (m < a.M)
          split_chunk_slot(v[r][m], sh[m], m, a.M, bcodes + (size_t)j * 2048, bsf + (size_t)j * 1024,
                           lane);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // read by tcgen05.mma / .cp
      __syncwarp();
      if (lane == 0) mbar_arrive(&cb.slot_ready[j]);
    }
  }
  // slots this call does not use: one arrival per call all the same
  if (lane == 0)
    for (int j = w; j < n_all; j += kChainSplitW)
      if (j >= a.n_slots) mbar_arrive(&cb.slot_ready[j]);
}

__global__ void __launch_bounds__(kThreads, 1) gemv_f4c_kernel(const __grid_constant__ F4Chain ch) {
  using L = StageR;
  constexpr int NMMA = 16;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t *bcodes = smem + kNSR * L::BYTES;              // [slot][16 rows][128 B], swizzled
  uint8_t *bsf = bcodes + (size_t)ch.n_slots * 2048;     // [slot][4 steps][256 B] + pad
  F4Bars &bars = *reinterpret_cast<F4Bars *>(bsf + (size_t)ch.n_slots * 1024 + 256);
  F4ChainBars &cb = *reinterpret_cast<F4ChainBars *>(reinterpret_cast<uint8_t *>(&bars) +
                                                     ((sizeof(F4Bars) + 15) & ~size_t(15)));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int32_t *status = ch.call[0].status;

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) {
    for (int j = 0; j < ch.n_slots; ++j) mbar_init(&cb.slot_ready[j], 1);
    init_common(bars, kNSR, kIssuersR);
  }
  if (warp == 0) tmem_alloc(&bars.tmem);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem;

  if (warp == kProducerR) {
    // Every call's weight in turn through one ring (position g -> slot
    // g % 8); the source of a stage is found before its slot frees.
    if (lane == 0) {
      int issued = 0;
      bool ok = true;
      for (int c = 0; c < ch.n_calls && ok; ++c) {
        const F4Args &a = ch.call[c];
        const StreamK sk(a.n_tiles, a.n_chunks, a.sched, a.ksplit, a.grid);
        PreparedTile src;
        for (int i = 0; i < sk.n_st; ++i) {
          int tile, chn;
          sk.tile_ch(sk.stage_of(i), tile, chn);
          src.at(a, tile, sk.nch);
          const uint8_t *w = src.wc + (size_t)chn * 16384, *sf = src.wsa + (size_t)chn * 2048;
          const int s = issued % kNSR;
          if (issued >= kNSR &&
              !mbar_wait_bounded(&bars.empty[s], (uint32_t)((issued / kNSR - 1) & 1), status)) {
            ok = false;
            break;
          }
          uint8_t *stg = smem + (size_t)s * L::BYTES;
          mbar_arrive_expect_tx(&bars.full[s], L::TX);
          bulk_g2s(stg + L::W, w, 16384u, &bars.full[s]);
          bulk_g2s(stg + L::SFA, sf, 2048u, &bars.full[s]);
          ++issued;
        }
      }
      // never leave with copies in flight
      for (int k = (issued > kNSR ? issued - kNSR : 0); k < issued; ++k)
        mbar_wait_bounded(&bars.full[k % kNSR], (uint32_t)((k / kNSR) & 1), status);
    }
  } else if (warp < kIssuersR) {
    const uint64_t dB0 = sdesc(smem_u32(bcodes), 16, 1024, kSw128);
    const uint64_t dSB0 = sdesc(smem_u32(bsf), 0, 128, kNoSwizzle);
    int ib = 0, jb = 0, n_splits = 0;
    bool ok = true;
    for (int c = 0; c < ch.n_calls && ok; ++c) {
      const F4Args &a = ch.call[c];
      const StreamK sk(a.n_tiles, a.n_chunks, a.sched, a.ksplit, a.grid);
      // a call that keeps the previous call's slots waits on the same phase
      if (!ch.reuse[c]) ++n_splits;
      const uint32_t par = (uint32_t)((n_splits - 1) & 1);
      // Wait for this call's split even with no stage in it: a parity wait
      // is only right one phase ahead, and an issuer that skipped calls
      // would otherwise take an older phase for this call's.  Every split
      // arrives on slot 0 after all warps finished the previous split, so
      // every slot barrier is at this call's phase or the one before.
      if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(&cb.slot_ready[0], par, status))) {
        ok = false;
        break;
      }
      auto b_desc = [&](int, int st, int t) {
        return dB0 + (uint64_t)((st % sk.nch) * (2048 >> 4)) + 2u * t;
      };
      auto sfb_desc = [&](int, int st, int t) {
        return dSB0 + (uint64_t)((st % sk.nch) * (1024 >> 4)) + (uint64_t)(16u * t);
      };
      auto b_wait = [&](int st) { return mbar_wait_bounded(&cb.slot_ready[st % sk.nch], par, status); };
      ok = issuer_loop<kIssuersR, kNSR, NMMA, true, L>(smem, bars, tmem, sk, warp, lane, status, b_desc,
                                                       sfb_desc, b_wait, ib, jb, true);
      ib += sk.n_st;
      jb += sk.n_seg;
    }
    issuer_drain(bars, warp, lane, status);
  } else if (warp == kLoaderWarpR || warp == kRelayWarp || warp == kSplitWarpX || warp >= kEpiWarp0) {
    // Split warps (5, 6, 7, 8..11); 8..11 also run the epilogue.  Per call:
    // wait for X if it is the previous call's output (one thread), meet
    // (every split warp, the epilogue warps after the previous call's
    // epilogue: its MMAs are complete, so the slots are free), split, then
    // the epilogue and this CTA's count for the call.
    const int w = warp < kEpiWarp0 ? warp - kLoaderWarpR : warp - kEpiWarp0 + 3;
    if (w == 0 && lane < 16)  // read (into lanes no N = 16 MMA uses) after the last slot
      reinterpret_cast<uint4 *>(bsf + (size_t)ch.n_slots * 1024)[lane] = make_uint4(0, 0, 0, 0);
    asm volatile("griddepcontrol.wait;" ::: "memory");  // X may come from the previous kernel
    if (blockIdx.x == 0 && w == 0) {
      // clear the counters (and the split-tile counts of stream-K calls),
      // then publish this launch (the previous launch on the stream has
      // finished: the wait above)
      for (int c = 0; c < ch.n_calls; ++c)
        if (ch.call[c].cnt32)
          for (int t = lane; t < ch.call[c].n_tiles; t += 32) ch.call[c].cnt32[t] = 0u;
      if (lane < kMaxChain) ch.cnt->done[lane] = 0u;
      if (lane == 0) ch.cnt->finished = 0u;
      __threadfence();
      __syncwarp();
      if (lane == 0)
        asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(&ch.cnt->ready), "l"(ch.epoch) : "memory");
    }
    // A thread checks that the counters are this launch's right before it
    // first counts or reads a count (by then CTA 0 has long published).
    bool ready_seen = false;
    int ib = 0, jb = 0, n_split = 0;
    bool ok = true;
    int sh[kMaxRowsX] = {};
    for (int c = 0; c < ch.n_calls; ++c) {
      const F4Args &a = ch.call[c];
      const StreamK sk(a.n_tiles, a.n_chunks, a.sched, a.ksplit, a.grid);
      if (!ch.reuse[c]) {
        if (c > 0 && ch.dep[c] && w == 0 && lane == 0) {
          if (!ready_seen) {
            chain_wait_ready(ch.cnt, ch.epoch, status);  // gives up (and reports) after 1 s
            ready_seen = true;
          }
          chain_wait_count(&ch.cnt->done[c - 1], gridDim.x, status);
        }
        asm volatile("bar.sync 1, %0;" ::"n"(32 * kChainSplitW) : "memory");
        chain_split(a, sk.ch0, sk.nch, ch.n_slots, w, lane, cb, bcodes, bsf, sh);
      }
      if (warp >= kEpiWarp0) {
        // the thread that counts split tiles and calls checks the counters
        // once (CTA 0 published them long before)
        if (c == 0 && warp == kEpiWarp0 && lane == 0) chain_wait_ready(ch.cnt, ch.epoch, status);
        if (ok) ok = epilogue_loop<kIssuersR, NMMA>(a, bars, tmem, sk, warp, lane, sh, nullptr, ib, jb, n_split);
        asm volatile("bar.sync 2, 128;" ::: "memory");
        if (warp == kEpiWarp0 && lane == 0) {
          __threadfence();  // this CTA's outputs of call c, then its count
          atomicAdd(&ch.cnt->done[c], 1u);
        }
      }
      ib += sk.n_st;
      jb += sk.n_seg;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_free(tmem);
  }
  // the last CTA to finish withdraws the launch (all others are past their
  // waits); the next launch's CTA 0 clears the counts
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(&ch.cnt->finished, 1u) == gridDim.x - 1) {
      __threadfence();
      ch.cnt->ready = 0ull;
    }
  }
}

// ---- host --------------------------------------------------------------------

// Operand rows: eight components per row of X, rounded up to an MMA width.
int nmma_for(int64_t M) { return M <= 2 ? 16 : M <= 4 ? 32 : M <= 8 ? 64 : 128; }

struct F4Ws {
  size_t bcodes, sfb, sh, cnt, part, total;
  int grid;  // streamed kernel: CTAs of its stream-K schedule
};
// Workspace of one call: X's components (the streamed kernel's codes
// [N_MMA][K/2] and atoms [K/64][512], or the resident kernel's slot images,
// codes [K/256][2 KB] -- the same size at N_MMA = 16 -- and scales
// [K/256][1 KB]), prescale exponents, per-tile counters, split-tile partials.
F4Ws f4_ws(int64_t M, int64_t N, int64_t K) {
  F4Ws w;
  const int nmma = nmma_for(M);
  const int64_t n_tiles = ceil_div(N, kTileRows);
  const int64_t chunks = n_tiles * (K / kChunkK);
  const int64_t cap = chunks < kMaxGrid ? chunks : kMaxGrid;
  w.grid = (int)(cap < num_sms() ? cap : num_sms());
  w.bcodes = 0;
  w.sfb = (size_t)ceil_div((int64_t)nmma * (K / 2), 1024) * 1024;
  w.sh = w.sfb + (size_t)(K / 64) * 512;
  w.cnt = w.sh + 256;
  w.part = w.cnt + (size_t)ceil_div(n_tiles * 16, 256) * 256;
  w.total = w.part + (size_t)cap * 2 * (nmma / kNC) * kTileRows * sizeof(float);
  return w;
}

template <int NMMA> size_t smem_s() {
  return (size_t)CfgS<NMMA>::NS * StageS<NMMA>::BYTES + sizeof(F4Bars) + 1024;
}

// The resident kernel's schedule for a shape (M <= 2):
//  * at least 3/4 as many tiles as SMs: whole tiles, as evenly as they
//    divide over at most one CTA per SM (no split-tile fix-ups, whose
//    global-memory round trips are slow while HBM is saturated; with fewer
//    tiles than SMs the SMs left over start the next kernel's weight stream
//    early);
//  * fewer: each tile's K split over a cluster of S = SMs / tiles CTAs
//    (at most 8, at most one chunk each), so that most SMs stream.
// n_slots: the most distinct K chunks a CTA sees (its B slots).
struct F4Plan {
  int sched, ksplit, grid, n_slots;
  bool split_inside;  // NVFP4: the kernel splits X itself (at most kSplitW slots)
  size_t smem;
  bool ok;  // the resident kernel takes the shape
};
F4Plan plan_r(int64_t M, int64_t N, int64_t K, int fmt = kFmtNv) {
  F4Plan p = {};
  const int chunk = fmt == kFmtF8 ? FmtR<kFmtF8>::kChunk : FmtR<kFmtNv>::kChunk;
  const int max_slots = fmt == kFmtF8 ? FmtR<kFmtF8>::kMaxSlots : FmtR<kFmtNv>::kMaxSlots;
  const uint32_t stage = fmt == kFmtF8 ? FmtR<kFmtF8>::kStageBytes : FmtR<kFmtNv>::kStageBytes;
  const uint32_t slot = 2048 + (fmt == kFmtF8 ? FmtR<kFmtF8>::kSlotSf : FmtR<kFmtNv>::kSlotSf);
  const int64_t nch = K / chunk, n_tiles = ceil_div(N, kTileRows), sms = num_sms();
  p.sched = kSchedStreamK;
  p.ksplit = 1;
  if (4 * n_tiles >= 3 * sms) {
    p.sched = kSchedWhole;
    p.grid = (int)(n_tiles < sms ? n_tiles : sms);
    p.n_slots = (int)nch;
  } else if (n_tiles < sms) {
    int64_t S = sms / n_tiles;
    if (S > 8) S = 8;
    if (S > nch) S = nch;
    if (S >= 2 && ceil_div(nch, S) <= max_slots) {
      p.sched = kSchedCluster;
      p.ksplit = (int)S;
      p.grid = (int)(n_tiles * S);
      p.n_slots = (int)ceil_div(nch, S);
    }
  }
  if (p.sched == kSchedStreamK || p.n_slots > max_slots) {
    p.sched = kSchedStreamK;
    p.ksplit = 1;
    int64_t g = n_tiles * nch;
    if (g > kMaxGrid) g = kMaxGrid;
    if (g > sms) g = sms;
    p.grid = (int)g;
    const int64_t per = ceil_div(n_tiles * nch, p.grid);
    p.n_slots = (int)(per < nch ? per : nch);
  }
  const size_t red = p.sched == kSchedCluster ? (size_t)(p.ksplit - 1) * kTileRows * 2 * sizeof(float) : 0;
  p.smem = (size_t)kNSR * stage + (size_t)p.n_slots * slot + 256 +
           ((sizeof(F4Bars) + 15) & ~size_t(15)) + red + 1024;
  // the split kernel stages a row of X (2 K bytes) in shared memory
  p.ok = M <= 2 && p.n_slots <= max_slots && K * 2 <= 200 * 1024 && p.smem <= 227 * 1024;
  p.split_inside = fmt == kFmtNv && p.n_slots <= kSplitW;
  if (p.split_inside) p.smem += sizeof(F4SplitBars);
  return p;
}

// Tensor maps cached per (array, shape).
struct MapEntry {
  const void *base;
  uint64_t rows, row_bytes;
  uint32_t box_rows, box_bytes;
  bool swz;
  CUtensorMap map;
};
std::mutex g_mu;
MapEntry g_cache[32];
int g_next = 0, g_used = 0;

bool cached_map(CUtensorMap &out, const void *base, uint64_t rows, uint64_t row_bytes,
                uint32_t box_rows, uint32_t box_bytes, bool swz) {
  std::lock_guard<std::mutex> lock(g_mu);
  for (int i = 0; i < g_used; ++i) {
    const MapEntry &e = g_cache[i];
    if (e.base == base && e.rows == rows && e.row_bytes == row_bytes && e.box_rows == box_rows &&
        e.box_bytes == box_bytes && e.swz == swz) {
      out = e.map;
      return true;
    }
  }
  if (!make_tmap_u8_2d(&out, base, rows, row_bytes, row_bytes, box_rows, box_bytes, swz))
    return false;
  MapEntry &e = g_cache[g_next];
  e = MapEntry{base, rows, row_bytes, box_rows, box_bytes, swz, out};
  g_next = (g_next + 1) % 32;
  if (g_used < 32) ++g_used;
  return true;
}

// Launch with programmatic dependent launch allowed, in clusters of
// `cluster` CTAs along x (1: no cluster).
template <class Kern, class... Args>
cudaError_t launch_pdl(Kern kern, int grid, int threads, size_t smem, cudaStream_t stream,
                       int cluster, Args... args) {
  if (smem > 48 * 1024) {
    const cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = (unsigned)cluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = cluster > 1 ? 2 : 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args...);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// 128-row tiles of all groups of a call
int64_t group_tiles(const GemvGroup *g, int n) {
  int64_t t = 0;
  for (int i = 0; i < n; ++i) t += ceil_div(g[i].N, kTileRows);
  return t;
}

F4Args base_args(const uint16_t *x, int64_t M, int64_t K, int64_t ldx, const GemvGroup *g, int n,
                 int32_t *status, uint8_t *ws, const F4Ws &L) {
  F4Args a = {};
  a.x = x;
  a.ldx = ldx;
  a.M = (int)M;
  a.K = K;
  a.sfb = ws + L.sfb;
  a.sh = reinterpret_cast<const int32_t *>(ws + L.sh);
  a.part = reinterpret_cast<float *>(ws + L.part);
  a.cnt = reinterpret_cast<unsigned __int128 *>(ws + L.cnt);
  a.status = status;
  a.n_groups = n;
  int64_t t = 0;
  for (int i = 0; i < n; ++i) {
    a.grp[i] = F4Group{g[i].codes, g[i].scales, g[i].tensor_scale, g[i].y, g[i].N, g[i].ldy, (int)t};
    t += ceil_div(g[i].N, kTileRows);
  }
  a.n_tiles = (int)t;
  a.n_chunks = (int)(K / kChunkK);
  a.epoch = next_launch_epoch();
  return a;
}

// Tensor maps of a row-major weight (a prepared weight is read with bulk
// copies: its maps stay zero and unread).
bool weight_maps(bool prepared, const uint8_t *codes, const uint8_t *scales, int64_t N, int64_t K,
                 CUtensorMap &mw, CUtensorMap &ms) {
  if (prepared) {
    memset(&mw, 0, sizeof(mw));
    memset(&ms, 0, sizeof(ms));
    return true;
  }
  return cached_map(mw, codes, (uint64_t)N, (uint64_t)(K / 2), kTileRows, 128, true) &&
         cached_map(ms, scales, (uint64_t)N, (uint64_t)(K / 16), kTileRows, 16, false);
}

// The streamed kernel's schedule, chosen as for the resident kernel: whole
// tiles with at least 3/4 as many tiles as SMs; fewer tiles: each tile's K
// split over a cluster of S CTAs whose partials meet in rank 0's shared
// memory (S limited by that buffer's room); otherwise stream-K.
struct SPlan {
  int sched, ksplit, grid;
  size_t smem;
};
template <int NMMA>
SPlan plan_s(int64_t N, int64_t K, int sk_grid) {
  SPlan p = {kSchedStreamK, 1, sk_grid, smem_s<NMMA>()};
  const int64_t nch = K / kChunkK, n_tiles = ceil_div(N, kTileRows), sms = num_sms();
  const size_t per_rank = (size_t)kTileRows * (NMMA / kNC) * sizeof(float);
  if (4 * n_tiles >= 3 * sms) {
    p.sched = kSchedWhole;
    p.grid = (int)(n_tiles < sms ? n_tiles : sms);
  } else if (n_tiles < sms) {
    int64_t S = sms / n_tiles;
    if (S > 8) S = 8;
    if (S > nch) S = nch;
    while (S >= 2 && smem_s<NMMA>() + (size_t)(S - 1) * per_rank > 227 * 1024) --S;
    if (S >= 2) {
      p.sched = kSchedCluster;
      p.ksplit = (int)S;
      p.grid = (int)(n_tiles * S);
      p.smem = smem_s<NMMA>() + (size_t)(S - 1) * per_rank;
    }
  }
  return p;
}

template <int NMMA>
cudaError_t launch_streamed(bool prepared, int sk_grid, cudaStream_t stream,
                            const CUtensorMap &mw, const CUtensorMap &ms, const CUtensorMap &mb,
                            F4Args a) {
  const SPlan P = plan_s<NMMA>(a.grp[0].N, a.K, sk_grid);
  a.sched = P.sched;
  a.ksplit = P.ksplit;
  const int cluster = P.sched == kSchedCluster ? P.ksplit : 1;
  return prepared ? launch_pdl(gemv_f4_kernel<NMMA, true>, P.grid, kThreads, P.smem, stream,
                               cluster, mw, ms, mb, a)
                  : launch_pdl(gemv_f4_kernel<NMMA, false>, P.grid, kThreads, P.smem, stream,
                               cluster, mw, ms, mb, a);
}

cudaError_t launch_pass_streamed(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                                 const uint8_t *codes, const uint8_t *scales,
                                 const float *tensor_scale, int64_t N, uint16_t *y, int64_t ldy,
                                 int32_t *status, void *workspace, cudaStream_t stream,
                                 bool prepared, const uint16_t *x2, int64_t ldx2) {
  const int nmma = nmma_for(M);
  const F4Ws L = f4_ws(M, N, K);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  CUtensorMap mw, ms, mb;
  if (!weight_maps(prepared, codes, scales, N, K, mw, ms) ||
      !cached_map(mb, ws + L.bcodes, (uint64_t)nmma, (uint64_t)(K / 2), (uint32_t)nmma, 128, true))
    return cudaErrorInvalidValue;
  // components of X (programmatic dependent launch: may start while the
  // previous kernel drains; it waits before reading X or writing the workspace)
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ceil_div(K / 16, kXsplitThreads), (unsigned)M);
    cfg.blockDim = dim3(kXsplitThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, xsplit_kernel, x, ldx, (int)M, K, nmma,
                                             ws + L.bcodes, ws + L.sfb,
                                             reinterpret_cast<int32_t *>(ws + L.sh), x2, ldx2);
    if (e != cudaSuccess) return e;
  }
  const GemvGroup g = {codes, scales, tensor_scale, y, N, ldy};
  F4Args a = base_args(x, M, K, ldx, &g, 1, status, ws, L);
  switch (nmma) {
    case 16: return launch_streamed<16>(prepared, L.grid, stream, mw, ms, mb, a);
    case 32: return launch_streamed<32>(prepared, L.grid, stream, mw, ms, mb, a);
    case 64: return launch_streamed<64>(prepared, L.grid, stream, mw, ms, mb, a);
    default: return launch_streamed<128>(prepared, L.grid, stream, mw, ms, mb, a);
  }
}

}  // namespace

unsigned long long next_launch_epoch() {
  static std::atomic<unsigned long long> epoch{0};
  static std::once_flag once;
  std::call_once(once, [] {
    std::random_device rd;
    epoch = ((unsigned long long)rd() << 32) ^ rd() ^
            (unsigned long long)std::chrono::steady_clock::now().time_since_epoch().count();
  });
  return ++epoch;
}

bool gemv_f4_shape_ok(int64_t M, int64_t N, int64_t K) {
  return M >= 1 && M <= kDecodeMaxM && N >= kTileRows && N <= 0x7FFFFFFFll && K >= 4 * kChunkK &&
         K % kChunkK == 0 && K <= (1 << 24);
}

size_t gemv_f4_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  return f4_ws(M, N, K).total;
}

int gemv_f4_launches(int64_t M, int64_t N, int64_t K, const char **kernel) {
  if (!gemv_f4_shape_ok(M, N, K)) return 0;
  const F4Plan P = plan_r(M, N, K);
  if (P.ok) {
    *kernel = "gemv_f4r_kernel";  // the GEMV, after a split kernel unless it splits X itself
    return P.split_inside ? 1 : 2;
  }
  *kernel = "gemv_f4_kernel";  // split kernel + GEMV
  return 2;
}

int gemv_f4_swiglu_launches(int64_t M, int64_t N, int64_t K, const char **kernel) {
  if (!gemv_f4_shape_ok(M, N, K)) return 0;
  *kernel = plan_r(M, N, K).ok ? "gemv_f4r_kernel" : "gemv_f4_kernel";
  return 2;  // the split kernel forms X from the two rows, then the weight stream
}

bool gemv_f4_supported(int64_t M, int64_t N, int64_t K, const void *codes, const void *scales) {
  return gemv_f4_shape_ok(M, N, K) && !(((uintptr_t)codes | (uintptr_t)scales) & 15u);
}

// One launch pair for every group: the split kernel, then the resident
// kernel over the groups' tiles (plan checked by the caller).
static cudaError_t launch_resident(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                            const GemvGroup *g, int n, int32_t *status, void *workspace,
                            cudaStream_t stream, bool prepared, const uint16_t *x2 = nullptr,
                            int64_t ldx2 = 0) {
  const int64_t rows = group_tiles(g, n) * kTileRows;
  const F4Plan P = plan_r(M, rows, K);
  const F4Ws L = f4_ws(M, rows, K);
  CUtensorMap mw, ms;
  if (!weight_maps(prepared, g[0].codes, g[0].scales, g[0].N, K, mw, ms)) return cudaErrorInvalidValue;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  F4Args a = base_args(x, M, K, ldx, g, n, status, ws, L);
  a.n_slots = P.n_slots;
  a.sched = P.sched;
  a.ksplit = P.ksplit;
  a.slot_codes = ws + L.bcodes;
  // an X made from two rows (x2) is split by the split kernel only
  const bool inside = P.split_inside && !x2;
  if (!inside) {
    // X -> B slot images by the split kernel (programmatic dependent launch:
    // it may start while the previous kernel drains and waits before reading
    // X or writing the workspace); each CTA then copies its slots in
    const size_t xs_bytes = (size_t)K * 2 * (x2 ? 2 : 1);  // the staged row(s)
    if (xs_bytes > 48 * 1024) {
      const cudaError_t e = cudaFuncSetAttribute(
          xsplit_slots_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)xs_bytes);
      if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ceil_div(K / kChunkK, kSplitWarps), (unsigned)M);
    cfg.blockDim = dim3(32 * kSplitWarps * (x2 ? 4 : 1));
    cfg.dynamicSmemBytes = xs_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, xsplit_slots_kernel, x, ldx, (int)M, K,
                                             ws + L.bcodes, ws + L.sfb,
                                             reinterpret_cast<int32_t *>(ws + L.sh), status, x2,
                                             ldx2);
    if (e != cudaSuccess) return e;
  }
  const int cluster = P.sched == kSchedCluster ? P.ksplit : 1;
  if (inside)
    return prepared ? launch_pdl(gemv_f4r_kernel<true, kFmtNv, true>, P.grid, kThreads, P.smem,
                                 stream, cluster, mw, ms, a)
                    : launch_pdl(gemv_f4r_kernel<false, kFmtNv, true>, P.grid, kThreads, P.smem,
                                 stream, cluster, mw, ms, a);
  return prepared ? launch_pdl(gemv_f4r_kernel<true>, P.grid, kThreads, P.smem, stream, cluster,
                               mw, ms, a)
                  : launch_pdl(gemv_f4r_kernel<false>, P.grid, kThreads, P.smem, stream, cluster,
                               mw, ms, a);
}

cudaError_t launch_gemv_f4(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                           const uint8_t *codes, const uint8_t *scales, const float *tensor_scale,
                           int64_t N, uint16_t *y, int64_t ldy, int32_t *status, void *workspace,
                           cudaStream_t stream, bool prepared, const uint16_t *x2,
                           int64_t ldx2) {
  if (plan_r(M, N, K).ok) {
    const GemvGroup g = {codes, scales, tensor_scale, y, N, ldy};
    return launch_resident(x, M, K, ldx, &g, 1, status, workspace, stream, prepared, x2, ldx2);
  }
  // every row of X in one stream of W
  return launch_pass_streamed(x, M, K, ldx, codes, scales, tensor_scale, N, y, ldy, status,
                              workspace, stream, prepared, x2, ldx2);
}

// ---- FP8-E4M3 weights ------------------------------------------------------------

namespace {
// Workspace of one FP8 call: slot images [K/128][2 KB] | prescale exponents |
// per-tile counters | stream-K partials.
struct F8Ws {
  size_t sh, cnt, part, total;
};
F8Ws f8_ws(int64_t N, int64_t K) {
  F8Ws w;
  const int64_t n_tiles = ceil_div(N, kTileRows);
  w.sh = (size_t)(K / 128) * 2048;
  w.cnt = w.sh + 256;
  w.part = w.cnt + (size_t)ceil_div(n_tiles * 16, 256) * 256;
  w.total = w.part + (size_t)kMaxGrid * 2 * 2 * kTileRows * sizeof(float);
  return w;
}
}  // namespace

bool gemv_fp8_shape_ok(int64_t M, int64_t N, int64_t K) {
  return M >= 1 && M <= kDecodeMaxM && N >= kTileRows && N <= 0x7FFFFFFFll && K >= 512 &&
         K % 128 == 0 && plan_r(2, N, K, kFmtF8).ok;
}

size_t gemv_fp8_workspace_bytes(int64_t N, int64_t K) { return f8_ws(N, K).total; }

int gemv_fp8_launches(int64_t M) { return 2 * (int)ceil_div(M, 2); }

cudaError_t launch_gemv_fp8(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                            const uint8_t *codes, const float *tensor_scale, int64_t N,
                            uint16_t *y, int64_t ldy, int32_t *status, void *workspace,
                            cudaStream_t stream) {
  const F8Ws L = f8_ws(N, K);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  CUtensorMap mw, ms;
  if (!cached_map(mw, codes, (uint64_t)N, (uint64_t)K, kTileRows, 128, true))
    return cudaErrorInvalidValue;
  memset(&ms, 0, sizeof(ms));
  const size_t xs_bytes = (size_t)K * 2;
  if (xs_bytes > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(
        xsplit_f8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)xs_bytes);
    if (e != cudaSuccess) return e;
  }
  // passes of up to two rows of X (8 operand rows each), one stream of W each
  for (int64_t m0 = 0; m0 < M; m0 += 2) {
    const int mp = (int)(M - m0 < 2 ? M - m0 : 2);
    const F4Plan P = plan_r(mp, N, K, kFmtF8);
    F4Args a = {};
    a.x = x + m0 * ldx;
    a.ldx = ldx;
    a.M = mp;
    a.K = K;
    a.sh = reinterpret_cast<const int32_t *>(ws + L.sh);
    a.part = reinterpret_cast<float *>(ws + L.part);
    a.cnt = reinterpret_cast<unsigned __int128 *>(ws + L.cnt);
    a.status = status;
    a.n_groups = 1;
    a.grp[0] = F4Group{codes, nullptr, tensor_scale, y + m0 * ldy, N, ldy, 0};
    a.n_tiles = (int)ceil_div(N, kTileRows);
    a.n_chunks = (int)(K / 128);
    a.epoch = next_launch_epoch();
    a.n_slots = P.n_slots;
    a.sched = P.sched;
    a.ksplit = P.ksplit;
    a.slot_codes = ws;
    {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)ceil_div(K / 128, kSplitWarps), (unsigned)mp);
      cfg.blockDim = dim3(32 * kSplitWarps);
      cfg.dynamicSmemBytes = xs_bytes;
      cfg.stream = stream;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[0].val.programmaticStreamSerializationAllowed = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      const cudaError_t e = cudaLaunchKernelEx(&cfg, xsplit_f8_kernel, a.x, ldx, mp, K, ws,
                                               reinterpret_cast<int32_t *>(ws + L.sh), status);
      if (e != cudaSuccess) return e;
    }
    const int cluster = P.sched == kSchedCluster ? P.ksplit : 1;
    const cudaError_t e = launch_pdl(gemv_f4r_kernel<false, kFmtF8>, P.grid, kThreads, P.smem,
                                     stream, cluster, mw, ms, a);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

bool gemv_f4_grouped_ok(int64_t M, int64_t K, const GemvGroup *g, int n) {
  if (n < 1 || n > kMaxGroups || M < 1 || M > 2 || K < 4 * kChunkK || K % kChunkK || K > (1 << 24))
    return false;
  for (int i = 0; i < n; ++i)
    if (g[i].N < 1 || g[i].N > 0x7FFFFFFFll || (((uintptr_t)g[i].codes | (uintptr_t)g[i].scales) & 15u))
      return false;
  const int64_t tiles = group_tiles(g, n);
  return tiles <= 0x7FFFFFFFll / kTileRows && plan_r(M, tiles * kTileRows, K).ok;
}

size_t gemv_f4_grouped_workspace_bytes(int64_t M, int64_t K, const int64_t *N, int n) {
  int64_t tiles = 0;
  for (int i = 0; i < n; ++i) tiles += ceil_div(N[i], kTileRows);
  return f4_ws(M, tiles * kTileRows, K).total;
}

cudaError_t launch_gemv_f4_grouped(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                                   const GemvGroup *g, int n, int32_t *status, void *workspace,
                                   cudaStream_t stream) {
  return launch_resident(x, M, K, ldx, g, n, status, workspace, stream, true);
}


// ---- chained calls ------------------------------------------------------------------

namespace {
// The chain's schedule: per link whole tiles (at least 3/4 as many tiles as
// SMs) or stream-K over all SMs, and its B slots; the workspace: the
// counters (256 bytes), then per stream-K link its tile counters and
// partial sums.
struct ChainPlan {
  int sched[kMaxChain], grid[kMaxChain], n_slots[kMaxChain], max_slots;
  size_t cnt[kMaxChain], part[kMaxChain], total, smem;
  bool ok;
};
ChainPlan plan_chain(int64_t M, const ChainLink *l, int n) {
  ChainPlan p = {};
  const int64_t G = num_sms();
  if (n < 1 || n > kMaxChain || M < 1 || M > 2 || G > kMaxGrid) return p;
  size_t off = 256;
  for (int c = 0; c < n; ++c) {
    const int64_t K = l[c].K;
    if (l[c].n < 1 || l[c].n > kMaxGroups || K < 4 * kChunkK || K % kChunkK || K > (1 << 24))
      return p;
    for (int i = 0; i < l[c].n; ++i) {
      const GemvGroup &g = l[c].g[i];
      if (g.N < 1 || g.N > 0x7FFFFFFFll || (((uintptr_t)g.codes | (uintptr_t)g.scales) & 15u))
        return p;
    }
    const int64_t tiles = group_tiles(l[c].g, l[c].n), nch = K / kChunkK;
    if (tiles * nch > 0x7FFFFFFFll) return p;
    if (4 * tiles >= 3 * G) {
      p.sched[c] = kSchedWhole;
      p.n_slots[c] = (int)nch;
    } else {
      p.sched[c] = kSchedStreamK;
      p.grid[c] = (int)(tiles * nch < G ? tiles * nch : G);
      const int64_t per = ceil_div(tiles * nch, p.grid[c]);
      p.n_slots[c] = (int)(per < nch ? per : nch);
      p.cnt[c] = off;
      off += (size_t)ceil_div(tiles * 16, 256) * 256;
      p.part[c] = off;
      off += (size_t)kMaxGrid * 2 * 2 * kTileRows * sizeof(float);
    }
    if (p.n_slots[c] > kChainSlots) return p;
    if (p.n_slots[c] > p.max_slots) p.max_slots = p.n_slots[c];
  }
  p.total = off;
  p.smem = (size_t)kNSR * StageR::BYTES + (size_t)p.max_slots * (2048 + 1024) + 256 +
           ((sizeof(F4Bars) + 15) & ~size_t(15)) + sizeof(F4ChainBars) + 1024;
  p.ok = p.smem <= 227 * 1024;
  return p;
}
}  // namespace

bool gemv_f4_chain_ok(int64_t M, const ChainLink *l, int n) { return plan_chain(M, l, n).ok; }

size_t gemv_f4_chain_workspace_bytes(int64_t M, const ChainLink *l, int n) {
  const ChainPlan P = plan_chain(M, l, n);
  return P.ok ? P.total : 0;
}

cudaError_t launch_gemv_f4_chain(int64_t M, const ChainLink *l, int n, int32_t *status,
                                 void *workspace, cudaStream_t stream) {
  const ChainPlan P = plan_chain(M, l, n);
  if (!P.ok) return cudaErrorInvalidValue;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  F4Chain ch = {};
  ch.n_calls = n;
  ch.n_slots = P.max_slots;
  ch.cnt = reinterpret_cast<ChainCounters *>(ws);
  ch.epoch = next_launch_epoch();
  for (int c = 0; c < n; ++c) {
    F4Args &a = ch.call[c];
    a.x = l[c].x;
    a.ldx = l[c].ldx;
    a.x2 = l[c].x2;
    a.ldx2 = l[c].ldx2;
    a.M = (int)M;
    a.K = l[c].K;
    a.status = status;
    if (P.sched[c] == kSchedStreamK) {
      a.cnt32 = reinterpret_cast<unsigned int *>(ws + P.cnt[c]);
      a.part = reinterpret_cast<float *>(ws + P.part[c]);
    }
    a.n_groups = l[c].n;
    int64_t t = 0;
    for (int i = 0; i < l[c].n; ++i) {
      const GemvGroup &g = l[c].g[i];
      a.grp[i] = F4Group{g.codes, g.scales, g.tensor_scale, g.y, g.N, g.ldy, (int)t};
      t += ceil_div(g.N, kTileRows);
    }
    a.n_tiles = (int)t;
    a.n_chunks = (int)(l[c].K / kChunkK);
    a.epoch = next_launch_epoch();
    a.n_slots = P.n_slots[c];
    a.sched = P.sched[c];
    a.grid = P.grid[c];
    a.ksplit = 1;
    ch.dep[c] = l[c].dep ? 1 : 0;
    // the previous call's B slots serve again: same X, same chunks in every
    // CTA (whole tiles: all of them), and not two such calls in a row (the
    // slot barriers' phases may run at most one call ahead of the issuers)
    ch.reuse[c] = c > 0 && !l[c].dep && !ch.reuse[c - 1] && l[c].x == l[c - 1].x &&
                  l[c].ldx == l[c - 1].ldx && l[c].K == l[c - 1].K && !l[c].x2 && !l[c - 1].x2 &&
                  P.sched[c] == kSchedWhole && P.sched[c - 1] == kSchedWhole;
  }
  cudaError_t e = cudaFuncSetAttribute(gemv_f4c_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)P.smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms());
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = P.smem;
  cfg.stream = stream;
  // The CTAs wait for each other, so all of them must be resident at once:
  // one per SM (its shared memory allows no second) and as many as SMs,
  // which holds whenever no other kernel occupies SMs for long (a wait gives
  // up after kWaitLimitNs and reports IMP_DEV_TIMEOUT).  A cooperative
  // launch would guarantee it but measured ~3.5 us slower per launch (it
  // gives up the overlap with the previous kernel).  Programmatic dependent
  // launch lets the weight stream start while the previous kernel drains.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, gemv_f4c_kernel, ch);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace impfp4
