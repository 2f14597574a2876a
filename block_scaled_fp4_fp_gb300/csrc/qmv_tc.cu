// qmv_tc.cu -- NVFP4 decode GEMV on the 5th-generation tensor cores.
//
// Pages: "epic: NVIDIA Volta (sm_70) inference acceleration program #1536"
// (Baseline: the decode step is the qmv weight stream; the V100 kernel is
// ALU-bound at 7.7 % of HBM), "mlx 0.30.7.3 -> 0.30.7.6" qqmm.cpp (the M = 1
// route: x against NVFP4 W stored [N, K]).
//
// The tensor core decodes the weights: W streams by TMA as the block-scaled
// FP4 A operand of tcgen05.mma.kind::mxf4nvf4 (E4M3 scales per 16, applied by
// the hardware), so no instruction touches a weight.  The bf16 activation x is
// written as kTerms = 6 FP4 terms in radix 8 over one power-of-two scale per
// CTA slice of K:
//     x = 2^e0 * (sum_t d_t 2^(6 - 3t) + r),   d_t in {-4, ..., 4},
// with max|x| / 2^e0 in [128, 256).  Rounding r_t 2^(3t-6) to the nearest
// integer and subtracting keeps every digit in [-4, 4]; term t stores d_t / 2
// (0, +-0.5, ..., +-2: exact e2m1 values) under the term scale 2^(7 - 3t)
// (2^7 ... 2^-8: exact E4M3 and E8M0 values), and |r| <= 2^-10, at most 2^-17
// of max|x|.  The terms are rows 0..5 of one 8-row B atom (rows 6, 7 hold zero
// codes; B rows 8..15 read an all-zero atom), so the term-scale tile is one
// constant tile.  The MMA yields D[row, t] = sum_k W[row, k] d_t[k] 2^(6-3t)
// in fp32 tensor memory; the epilogue forms y = gs_w 2^e0 sum_t D[row, t].
//
// Work split.  A cluster of `split` CTAs owns R <= 128 consecutive rows; CTA
// rank i of the cluster takes the i-th slice of the K stages (K = 256 each),
// so a light problem runs fewer, fuller stages per CTA.  Each CTA sums its
// slice into fp32 partials; ranks 1.. store theirs into rank 0's shared
// memory with asynchronous remote stores (distributed shared memory) that a
// barrier there counts by bytes, and rank 0 adds them in rank order -- the
// same order on every run -- and writes y.
//   warp 0: barrier setup (one barrier per lane), then the TMA producer: per
//           stage one box of R rows x 128 bytes of W (128-byte swizzle, so
//           rows land as the 8-row atoms the MMA reads) and one box of R rows
//           x 16 bytes of W's linear E4M3 scales, into a ring sized in bytes
//           (a slot holds ceil(R/8) KB of codes; about 128 KB, at least kMeta
//           slots, in flight).  Issued before griddepcontrol.wait (programmatic
//           dependent launch: W is not written by the kernel this one
//           overlaps);
//   warp 1: tensor memory allocation; one thread issues each stage's
//           4 MMAs (M 128, N 16, K 64) into four independent accumulators,
//           then one commit that frees the stage's operands.  A-operand rows
//           >= R read whatever follows the slot; their scales are zero;
//   warps 2-17: four groups of four warps (one per tensor-memory lane
//           quadrant); group g prepares local stages i % 4 == g into a ring of
//           kMeta operand slots: the x terms in shared memory, then, once the
//           stage's weights have landed, each thread stores its row's 16
//           scale bytes straight into the slot's scale columns of tensor
//           memory (tcgen05.st).  A group that finds operand slot m free again
//           (stage i - kMeta done) passes the weight slot of that stage back
//           to the TMA producer.  After the last stage group 0 reads D and
//           forms the partials.
#include <algorithm>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace fp4 {

namespace {

constexpr int kTerms = 6;           // x expansion terms (B rows 0..5)
constexpr int kMetaMax = 6;         // ring of per-stage MMA operands built by the prep warps, at most
constexpr int kMaxSlots = 32;       // weight ring slots at most
constexpr uint32_t kInflightBytes = 128u * 1024u;  // weight bytes a CTA keeps in flight at most
constexpr int kChunk = 256;         // codes per TMA box (128 bytes per row)
constexpr int kRows = 128;          // rows per CTA at most (one M = 128 tile)
constexpr int kMaxSplit = 8;        // CTAs per cluster at most (portable cluster size)
constexpr int kGroups = 4;          // prep groups; group g prepares local stages i % kGroups == g
constexpr int kGroupThreads = 128;  // one group = 4 warps, two elements per thread per stage
constexpr int kPrep = kGroups * kGroupThreads;
constexpr int kThreads = 64 + kPrep;  // TMA warp, MMA warp, prep warps (group 0 also runs the epilogue)
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kSfbCol = 64;         // D: four accumulators of 16 columns in [0, 64); term scales
constexpr uint32_t kSfaCol = 80;         // weight scales of operand slot m: kSfaCol + 16 m + 4 j
static_assert(kMaxSlots <= 32 && kMetaMax <= 32, "one barrier pair per lane of warp 0");
// kind::mxf4nvf4 descriptor: E2M1 A/B, K-major, N = 16, M = 128; bit 23 selects E8M0 scales
constexpr uint32_t kIdesc = (1u << 7) | (1u << 10) | ((16u >> 3) << 17) | ((128u >> 4) << 24);

// Per format: a stage is kCh chunks of 256 elements; a row carries kSB scale
// bytes per stage, which tcgen05.cp moves as kSB / 4 tiles of 128x4 scales.
// NVFP4 (E4M3 per 16): k-step j (K = 64) reads tile j; MXFP4 (E8M0 per 32):
// half j & 1 of tile j / 2, through the scale-factor id.
template <int MODE> struct Fmt;
template <> struct Fmt<2> {
  static constexpr int kCh = 1;
  static constexpr int kMeta = 6;   // operand ring depth
  static constexpr int kGroup = 16;
  static constexpr uint32_t kIdesc = fp4::kIdesc;
  // E4M3 byte of the term scale 2^(7-3t) (exact: 2^7 ... 2^-8, the last one subnormal)
  __host__ __device__ static constexpr uint32_t term_scale(int t) {
    return (7 - 3 * t >= -6) ? (uint32_t)((7 - 3 * t + 7) << 3) : (1u << (7 - 3 * t + 9));
  }
};
template <> struct Fmt<1> {
  static constexpr int kCh = 2;
  static constexpr int kMeta = 4;   // stages are twice as large: a shallower ring keeps kMeta weight slots
  static constexpr int kGroup = 32;
  static constexpr uint32_t kIdesc = fp4::kIdesc | (1u << 23);
  // E8M0 byte of 2^(7-3t)
  __host__ __device__ static constexpr uint32_t term_scale(int t) { return (uint32_t)(127 + 7 - 3 * t); }
};
template <int MODE> struct Geo {
  static constexpr int kCh = Fmt<MODE>::kCh;
  static constexpr int kMeta = Fmt<MODE>::kMeta;
  static constexpr int kBK = 256 * kCh;                          // codes per stage
  static constexpr int kSB = kBK / Fmt<MODE>::kGroup;             // scale bytes per row per stage
  static constexpr int kTiles = kSB / 4;                         // 128x4 scale tiles per stage
  static constexpr int kSpk = 64 / Fmt<MODE>::kGroup;             // scales per row per k-step
  static_assert(kSB == 16, "a row brings one 16-byte word of scales per stage: four scale tiles");
  static_assert(kSfaCol + kMeta * kTiles * 4 <= kTmemCols, "scale columns exceed the allocation");
};

// Shared memory (from a 1024-aligned base): [weight ring | term atoms | zero
// atom | term-scale tile | x slice | partials | barriers].
// The weight ring is split at launch into code slots and, after them, scale slots.
constexpr int kMaxKSlice = 17408;  // elements of x per CTA
constexpr uint32_t kSmemBytes = 227u * 1024u;
constexpr uint32_t kBarBytes = 1024;
constexpr uint32_t kRedBytes = kMaxSplit * kRows * 4;
template <int MODE> struct Lay {
  using G = Geo<MODE>;
  static_assert(G::kMeta >= kGroups && G::kMeta <= kMetaMax, "a group's stages must not share an operand slot");
  static constexpr uint32_t kAtoms = G::kMeta * G::kCh;  // term atoms in the operand ring (kCh per slot)
  static constexpr uint32_t kFixed = (kAtoms + 1) * 1024 + 512 + kMaxKSlice * 2 + kRedBytes + kBarBytes + 1024;
  static constexpr uint32_t kRing = (kSmemBytes - kFixed) / 1024u * 1024u;
  static constexpr uint32_t kOffB = kRing;                  // B rows 0..7 (terms, 2 zero rows): atom kCh m + h of slot m
  static constexpr uint32_t kOffZ = kOffB + kAtoms * 1024;  // B rows 8..15 of every stage: zero codes
  static constexpr uint32_t kOffSFB = kOffZ + 1024;
  static constexpr uint32_t kOffX = kOffSFB + 512;             // x slice (bf16)
  static constexpr uint32_t kOffRed = kOffX + kMaxKSlice * 2;  // [split][128] fp32 partials (rank 0)
  static constexpr uint32_t kOffBar = kOffRed + kRedBytes;
  static_assert(kOffBar + kBarBytes + 1024 <= kSmemBytes, "shared memory layout overflows");
  // an MMA reads 16 KB of A from a code chunk's start: that stays inside the allocation
  static_assert(kRing + 16384 <= kOffBar, "A-operand reads past the allocation");
};
static_assert((2 * kMaxSlots + 2 * kMetaMax + 5) * 8 + 16 + (kPrep / 32) * 4 <= kBarBytes, "barrier area");

__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(sbo >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
__device__ __forceinline__ uint64_t desc_sf(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(128 >> 4) << 32) | ((uint64_t)1 << 46);
}
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
// shared::cluster address of the same shared-memory location in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t map_rank(const void* p, int rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) qmv_tc_kernel(const __grid_constant__ CUtensorMap tmW,
                                                              const __grid_constant__ CUtensorMap tmS,
                                                              const uint16_t* __restrict__ x,
                                                              const float* __restrict__ gs_w, int N, int K,
                                                              int R, int split, int nslots, uint32_t wslot,
                                                              uint32_t sslot, uint16_t* __restrict__ y,
                                                              unsigned* __restrict__ err, int inject_timeout) {
  using F = Fmt<MODE>;
  using G = Geo<MODE>;
  using L = Lay<MODE>;
  constexpr int kCh = G::kCh;
  constexpr int kMeta = G::kMeta;
  constexpr int kBK = G::kBK;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  uint64_t* wfull = reinterpret_cast<uint64_t*>(smem + L::kOffBar);  // weight slot landed (TMA bytes)
  uint64_t* wempty = wfull + kMaxSlots;                           // weight slot consumed (relayed)
  uint64_t* mfull = wempty + kMaxSlots;                           // stage operands built (prep group)
  uint64_t* mempty = mfull + kMetaMax;                            // stage operands consumed (MMA commit)
  uint64_t* done = mempty + kMetaMax;
  uint64_t* xbar = done + 1;
  uint64_t* pbar = xbar + 1;  // rank 0: the other ranks' partials have landed (byte count)
  uint64_t* tbar = pbar + 1;  // warp 1 has allocated tensor memory (tmem_slot written)
  uint64_t* never = tbar + 1; // fault injection: a barrier nothing arrives at
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(never + 1);
  uint32_t* red = tmem_slot + 4;  // kPrep / 32 warp maxima of |x| (bf16 bits)
  float* part = reinterpret_cast<float*>(smem + L::kOffRed);
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem + L::kOffX);
  const uint32_t offS = (uint32_t)nslots * wslot;  // linear-scale slots follow the code slots
  const uint32_t wchunk = wslot / kCh;              // one 256-element chunk of a code slot

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = (int)(blockIdx.x % (unsigned)split);  // rank within the cluster (clusters are consecutive)
  const int blk = (int)(blockIdx.x / (unsigned)split);
  const int nblk = (int)(gridDim.x / (unsigned)split);
  const int r0 = (int)(((int64_t)N * blk) / nblk);
  const int r1 = (int)(((int64_t)N * (blk + 1)) / nblk);
  const int rows = r1 - r0;  // <= R <= 128
  const int nkb = K / kBK;
  const int kb0 = (int)(((int64_t)nkb * rank) / split);
  const int nst = (int)(((int64_t)nkb * (rank + 1)) / split) - kb0;  // this CTA's stages (>= 1)

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (warp == 0) {  // one barrier (pair) per lane
    if (lane < nslots) {
      mbar_init(&wfull[lane], 1);
      mbar_init(&wempty[lane], 1);
    }
    if (lane < kMeta) {
      mbar_init(&mfull[lane], kGroupThreads);
      mbar_init(&mempty[lane], 1);
    }
    if (lane == 0) {
      mbar_init(done, 1);
      mbar_init(xbar, 1);
      mbar_init(pbar, 1);
      mbar_init(tbar, 1);
      mbar_init(never, 1);
    }
    fence_barrier_init();  // release of the barrier inits to the cluster
  }
  // Ranks > 0 wait on this arrival before storing into rank 0's shared memory:
  // rank 0 has started and its barriers are initialized.
  __syncwarp();
  if (split > 1) cluster_arrive_relaxed();
  // The constant term-scale tile: B row t < 9 (tile row t, slot 0) holds the
  // E4M3 weight 2^(7-2t) for each of the k-step's four 16-element blocks;
  // rows 9..31 are zero, so B rows 9..15 add nothing.
  if (threadIdx.x < 128) {
    const int row = threadIdx.x >> 2, word = threadIdx.x & 3;
    const uint32_t v = (row < kTerms && word == 0) ? F::term_scale(row) * 0x01010101u : 0u;
    reinterpret_cast<uint32_t*>(smem + L::kOffSFB)[threadIdx.x] = v;
  }
  // zero codes: rows 6, 7 (bytes 768..1023) of every term atom, and the zero atom
  for (uint32_t i = threadIdx.x; i < L::kAtoms * 64 + 256; i += kThreads) {
    const uint32_t off = i < L::kAtoms * 64 ? (i >> 6) * 1024 + 768 + (i & 63) * 4 : L::kAtoms * 1024 + (i - L::kAtoms * 64) * 4;
    *reinterpret_cast<uint32_t*>(smem + L::kOffB + off) = 0u;
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncthreads();
  uint32_t tmem = 0;  // tensor-memory base: warp 1 after its allocation, group 0 after `done`
  bool failed = false;
  float partial = 0.f;  // group 0: this CTA's partial y of row 32 (warp & 3) + lane

  if (warp == 0) {
    // ------------------------------------------------ TMA producer (weights)
    if (elect_one_sync()) {
      prefetch_tmap(&tmW);
      prefetch_tmap(&tmS);
      // out-of-range rows are zero-filled and counted
      const uint32_t tx = (uint32_t)R * (128u * kCh + G::kSB);
      int s = 0, round = 0;
      for (int i = 0; i < nst; ++i) {
        if (round > 0) mbar_wait(&wempty[s], (round - 1) & 1, err, failed);
        mbar_arrive_expect_tx(&wfull[s], tx);
#pragma unroll
        for (int h = 0; h < kCh; ++h)
          tma_load_2d(smem + s * wslot + h * wchunk, &tmW, &wfull[s], ((kb0 + i) * kCh + h) * 128, r0);
        tma_load_2d(smem + offS + s * sslot, &tmS, &wfull[s], (kb0 + i) * G::kSB, r0);
        if (++s == nslots) { s = 0; ++round; }
      }
      // no copy may still be writing shared memory when the CTA exits
      for (int i = max(0, nst - nslots); i < nst; ++i)
        mbar_wait(&wfull[i % nslots], (i / nslots) & 1, err, failed);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    // The tensor-memory allocation takes about a microsecond: it happens here,
    // while the weights stream and the prep warps build the first operands.
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(tmem_slot)), "r"(kTmemCols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    tc_fence_before();
    __syncwarp();
    tc_fence_after();
    tmem = *tmem_slot;
    if (lane == 0) mbar_arrive(tbar);  // releases the tmem_slot write to the epilogue
    if (elect_one_sync()) {
      if (inject_timeout) {
        bool injected = false;  // separate flag: the injected expiry must not stop later waits
        mbar_wait(never, 0, err, injected, 2000000LL);
      }
      asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;"
                   :: "r"(tmem + kSfbCol), "l"(desc_sf(base + L::kOffSFB)) : "memory");
      const uint32_t sfb_t = tmem + kSfbCol;
      int m = 0, mround = 0, s = 0;
      for (int i = 0; i < nst; ++i) {
        mbar_wait(&mfull[m], mround & 1, err, failed);  // the group also saw the weights land
        tc_fence_after();
        const uint32_t sfa_t = tmem + kSfaCol + 4 * G::kTiles * m;  // 4-column aligned tiles
#pragma unroll
        for (int j = 0; j < 4 * kCh; ++j) {
          // k-step j (K = 64): chunk h = j / 4, 32 bytes further per k-step along the swizzled rows
          const int h = j >> 2, jj = j & 3;
          const uint64_t adesc = desc_sw128(base + s * wslot + h * wchunk, 1024) + (uint64_t)(2 * jj);
          // B rows 0..7: the chunk's term atom; rows 8..15: the zero atom
          const uint32_t batom = L::kOffB + (uint32_t)(m * kCh + h) * 1024;
          const uint64_t bdesc = desc_sw128(base + batom, L::kOffZ - batom) + (uint64_t)(2 * jj);
          // scale columns j kSpk .. of the stage: tile (j kSpk) / 4, scale-factor id (j kSpk) % 4
          const uint32_t tile = (uint32_t)((j * G::kSpk) >> 2);
          const uint32_t sf_id = (uint32_t)((j * G::kSpk) & 3);
          const uint32_t idesc = F::kIdesc | (sf_id << 29) | (sf_id << 4);
          // k-step j accumulates into tile j % 4 of D, so consecutive MMAs of a stage do
          // not wait on each other; the epilogue adds the four tiles
          const uint32_t acc = (i > 0 || j >= 4) ? 1u : 0u;
          if (MODE == 2)
            asm volatile(
                "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %6, 0;\n\t"
                "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
                :: "r"(tmem + 16 * (j & 3)), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_t + 4 * tile), "r"(sfb_t),
                   "r"(acc) : "memory");
          else
            asm volatile(
                "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %6, 0;\n\t"
                "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
                :: "r"(tmem + 16 * (j & 3)), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_t + 4 * tile), "r"(sfb_t),
                   "r"(acc) : "memory");
        }
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                     :: "r"(smem_u32(&mempty[m])) : "memory");
        if (++m == kMeta) { m = 0; ++mround; }
        if (++s == nslots) s = 0;
      }
      asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                   :: "r"(smem_u32(done)) : "memory");
    }
  } else {
    // ------------------------------------------- prep warps (2..17), then epilogue
    const int pa = threadIdx.x - 64;           // 0..kPrep-1
    const int grp = pa / kGroupThreads;        // prep group
    const int pt = pa % kGroupThreads;         // thread within the group
    if (split > 1 && rank > 0) cluster_wait();  // (see the arrival after the barrier inits)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // this CTA's slice of x (bf16, nst * 512 bytes) -> shared memory in one bulk copy
    const uint32_t xbytes = (uint32_t)nst * (kBK * 2);
    if (pa == 0) {
      mbar_arrive_expect_tx(xbar, xbytes);
      bulk_load(xs, x + (int64_t)kb0 * kBK, xbytes, xbar);
    }
    mbar_wait(xbar, 0, err, failed);
    uint32_t m2 = 0;
    for (int v = pa; v < nst * (kBK / 8); v += kPrep) {
      const uint4 q = reinterpret_cast<const uint4*>(xs)[v];
      m2 = __vmaxu2(m2, q.x & 0x7FFF7FFFu);
      m2 = __vmaxu2(m2, q.y & 0x7FFF7FFFu);
      m2 = __vmaxu2(m2, q.z & 0x7FFF7FFFu);
      m2 = __vmaxu2(m2, q.w & 0x7FFF7FFFu);
    }
    const uint32_t mb = __reduce_max_sync(0xffffffffu, max(m2 & 0xFFFFu, m2 >> 16));
    if (lane == 0) red[pa >> 5] = mb;
    asm volatile("bar.sync 1, %0;" :: "n"(kPrep) : "memory");  // prep warps only
    uint32_t mball = 0;
#pragma unroll
    for (int i = 0; i < kPrep / 32; ++i) mball = max(mball, red[i]);
    const float amax = __uint_as_float(mball << 16);
    // e0: max|x| / 2^e0 in [128, 256) (bf16 magnitudes sort as integers; a NaN
    // or infinity in the slice shows as a value above the largest finite one)
    const bool finite = amax <= 3.3895313892515355e38f;
    int e0 = 0;
    if (amax > 0.f && finite) {
      int ex;
      frexpf(amax, &ex);  // amax = m * 2^ex, 0.5 <= m < 1
      e0 = max(ex - 8, -126);
    }
    const float pre = ldexpf(1.0f, -e0);

    // tensor memory (warp 1 allocated it at the start): this warp's lane quadrant
    mbar_wait(tbar, 0, err, failed);
    tc_fence_after();
    const int srow = 32 * (warp & 3) + lane;  // the weight row whose scales this thread moves
    const uint32_t tmem_lane = *tmem_slot + ((uint32_t)(32 * (warp & 3)) << 16);
    // stage bookkeeping without divisions: operand slot m (round mr), weight slot s (round wr)
    int m = grp, mr = 0, s = grp, wr = 0;
    const int lo = pt & 15, hi4 = ((pt >> 4) & 7) << 4;
    for (int i = grp; i < nst; i += kGroups) {
      if (i >= kMeta) {
        mbar_wait(&mempty[m], (mr - 1) & 1, err, failed);  // operand slot m is free: stage i - kMeta is done
        tc_fence_after();  // its MMAs have read the slot's scale columns
        if (pt == 0) {
          int sj = s - kMeta;  // weight slot of stage i - kMeta (nslots >= kMeta)
          if (sj < 0) sj += nslots;
          mbar_arrive(&wempty[sj]);
        }
      }
      // (a) x terms for elements 256 h + 2pt, + 1 of this stage (radix-8 digits, see the header)
#pragma unroll
      for (int h = 0; h < kCh; ++h) {
        const uint32_t xv = *reinterpret_cast<const uint32_t*>(xs + i * kBK + h * kChunk + 2 * pt);
        float r0v = bf16_lo(xv) * pre, r1v = bf16_hi(xv) * pre;
        uint8_t* batom = smem + L::kOffB + (m * kCh + h) * 1024;
#pragma unroll
        for (int t = 0; t < kTerms; ++t) {
          // v = d / 2 with d = rint(r / 2^(6-3t)): one fused multiply-add onto 1.5 * 2^22
          // rounds the exact product r 2^(3t-7) to a multiple of 1/2 (ties to even d);
          // subtracting the constant back is exact
          const float inv = __int_as_float((127 + 3 * t - 7) << 23);  // 2^(3t-7)
          const float w = __int_as_float((127 + 7 - 3 * t) << 23);    // 2^(7-3t), the term scale
          const float v0 = __fsub_rn(__fmaf_rn(r0v, inv, 6291456.0f), 6291456.0f);
          const float v1 = __fsub_rn(__fmaf_rn(r1v, inv, 6291456.0f), 6291456.0f);
          r0v = __fmaf_rn(-w, v0, r0v);  // exact: |result| <= 2^(6-3t) / 2
          r1v = __fmaf_rn(-w, v1, r1v);
          const uint8_t code = (uint8_t)e2m1x2_rn(v0, v1);  // exact: v in {0, +-0.5, ..., +-2}
          // byte pt of term row t, 128-byte swizzle
          batom[t * 128 + ((hi4 ^ (t << 4))) + lo] = code;
        }
      }
      // (b) weight scales of row srow, once the stage has landed: its 16 scale bytes,
      // word j -> the four tensor-memory columns of scale tile j of operand slot m (the
      // MMA reads the column of this lane's quadrant; every one holds the row's
      // scales).  Rows >= rows get 0.
      mbar_wait(&wfull[s], wr & 1, err, failed);
      uint4 sv = make_uint4(0, 0, 0, 0);
      if (srow < rows) sv = *reinterpret_cast<const uint4*>(smem + offS + s * sslot + srow * G::kSB);
      asm volatile(
          "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %1, %1, %1, %2, %2, %2, %2, %3, %3, %3, %3, %4, %4, %4, %4};"
          :: "r"(tmem_lane + kSfaCol + 4 * G::kTiles * m), "r"(sv.x), "r"(sv.y), "r"(sv.z), "r"(sv.w) : "memory");
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      tc_fence_before();
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the term bytes, for the MMA
      mbar_arrive(&mfull[m]);
      m += kGroups;
      if (m >= kMeta) { m -= kMeta; ++mr; }
      s += kGroups;
      if (s >= nslots) { s -= nslots; ++wr; }
    }
    // ---- epilogue (group 0, warps 2..5 = lane quadrants 2, 3, 0, 1): partial = 2^e0 sum_t D[row, t]
    if (grp == 0) {
      mbar_wait(tbar, 0, err, failed);
      mbar_wait(done, 0, err, failed);
      tc_fence_after();
      tmem = *tmem_slot;
      const int q = warp & 3;
      // columns 0..7 of the four accumulators (terms 0..5, two zero columns)
      uint32_t d[4][8];
#pragma unroll
      for (int a = 0; a < 4; ++a)
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
            : "=r"(d[a][0]), "=r"(d[a][1]), "=r"(d[a][2]), "=r"(d[a][3]), "=r"(d[a][4]), "=r"(d[a][5]),
              "=r"(d[a][6]), "=r"(d[a][7])
            : "r"(tmem + ((uint32_t)(32 * q) << 16) + 16 * a));
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
      float dsum[kTerms];
#pragma unroll
      for (int t = 0; t < kTerms; ++t)
        dsum[t] = (__uint_as_float(d[0][t]) + __uint_as_float(d[1][t])) +
                  (__uint_as_float(d[2][t]) + __uint_as_float(d[3][t]));
      float acc = 0.f;
#pragma unroll
      for (int t = kTerms - 1; t >= 0; --t) acc += dsum[t];
      partial = finite ? ldexpf(acc, e0) : __int_as_float(0x7FC00000);
      const int row = 32 * q + lane;
      if (rank > 0) {
        // asynchronous store into rank 0's partials; its barrier counts the bytes
        if (row < rows)
          asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];"
                       :: "r"(map_rank(part + rank * kRows + row, 0)), "r"(__float_as_uint(partial)),
                          "r"(map_rank(pbar, 0)) : "memory");
      } else {
        if (split > 1) {
          if (pa == 0) mbar_arrive_expect_tx(pbar, (uint32_t)(split - 1) * (uint32_t)rows * 4u);
          mbar_wait(pbar, 0, err, failed);  // every other rank's partials have landed
        }
        if (row < rows) {
          float acc_y = partial;
          for (int c = 1; c < split; ++c) acc_y += part[c * kRows + row];
          const float g = gs_w ? __ldg(gs_w) : 1.0f;
          y[r0 + row] = (uint16_t)f32_to_bf16_rn(acc_y * g);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(kTmemCols) : "memory");
  }
}

// How many clusters of `split` CTAs of this kernel can be resident at once on
// the device (cached per device, format and split; 0 if the query fails).
template <int MODE>
int max_clusters(const DevInfo& d, int split) {
  static std::mutex mu;
  static int cache[64][kMaxSplit + 1];
  static bool have[64][kMaxSplit + 1];
  if (d.device < 0 || d.device >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (have[d.device][split]) return cache[d.device][split];
  int n = 0;
  if (cudaFuncSetAttribute(qmv_tc_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) ==
      cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(split * std::max(1, d.sm_count / split)));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)split;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, qmv_tc_kernel<MODE>, &cfg) != cudaSuccess) {
      n = 0;
      cudaGetLastError();  // the failed query leaves no sticky error behind
    }
  }
  cache[d.device][split] = n;
  have[d.device][split] = true;
  return n;
}

struct TcPlan {
  int split = 0;       // CTAs per cluster (K slices); 0 = no plan
  int nblk = 0;        // row blocks (clusters)
  int R = 0;           // rows per CTA at most (blocks own R or R - 1 rows)
  int nslots = 0;      // weight ring slots
  uint32_t wslot = 0;  // bytes of codes per slot (kCh chunks of ceil(R/8) swizzle atoms)
  uint32_t sslot = 0;  // bytes of linear scales per slot
};

// Choose the K split: per CTA the time is about (stages) x max(fixed issue cost
// of a stage, the stage's bytes at an even share of HBM bandwidth); the split
// with the smallest estimate wins (ties go to the smaller split).
template <int MODE>
TcPlan plan_qmv_tc(const DevInfo& d, int64_t N, int64_t K) {
  using G = Geo<MODE>;
  constexpr int kCh = G::kCh;
  constexpr int kMeta = G::kMeta;
  constexpr int kBK = G::kBK;
  TcPlan best;
  if (K % kBK != 0 || N < 1 || d.sm_count < 1) return best;
  const int64_t nkb = K / kBK;
  const double stage_us = 0.2 * kCh, sm_gbs = 43.0;
  double best_cost = 0.0;
  for (int split = 1; split <= kMaxSplit; ++split) {
    if (nkb < split) break;
    const int64_t nst = (nkb + split - 1) / split;
    if (nst * kBK > kMaxKSlice) continue;
    int64_t nblk = split == 1 ? d.sm_count : std::min<int64_t>(max_clusters<MODE>(d, split), d.sm_count / split);
    nblk = std::min<int64_t>(nblk, N);
    if (nblk < 1) continue;
    const int64_t R = (N + nblk - 1) / nblk;
    if (R > kRows) continue;
    const double cost = (double)nst * std::max(stage_us, (double)R * (128.0 * kCh + G::kSB) / (sm_gbs * 1e3));
    if (best.split == 0 || cost < best_cost) {
      best_cost = cost;
      best.split = split;
      best.nblk = (int)nblk;
      best.R = (int)R;
    }
  }
  if (best.split == 0) return best;
  best.wslot = (uint32_t)kCh * (uint32_t)((best.R + 7) / 8) * 1024u;
  best.sslot = ((uint32_t)best.R * G::kSB + 127u) / 128u * 128u;
  // deeper than about 128 KB only lengthens the queues in front of the first stages
  const uint32_t slot = best.wslot + best.sslot;
  best.nslots = (int)std::min<uint32_t>(kMaxSlots, Lay<MODE>::kRing / slot);
  best.nslots = std::max<int>(std::min<int>(best.nslots, kMeta), std::min<int>(best.nslots, kInflightBytes / slot));
  if (best.nslots < kMeta) best.split = 0;  // the slot relay needs nslots >= kMeta
  return best;
}

template <int MODE>
cudaError_t launch_mode_tc(const DevInfo& d, const uint16_t* x, const uint32_t* w, const uint8_t* scales,
                           const float* gs_w, int64_t N, int64_t K, uint16_t* y, int inject, cudaStream_t s) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorInvalidValue;
  const TcPlan p = plan_qmv_tc<MODE>(d, N, K);
  if (p.split == 0) return cudaErrorInvalidValue;
  const int group = MODE == 2 ? 16 : 32;
  cuuint32_t estr[2] = {1, 1};
  // W codes: [N, K/2] bytes, boxes of R rows x 128 bytes, 128-byte swizzle
  CUtensorMap tmW;
  {
    cuuint64_t dims[2] = {(cuuint64_t)(K / 2), (cuuint64_t)N};
    cuuint64_t strides[1] = {(cuuint64_t)(K / 2)};
    cuuint32_t box[2] = {128, (cuuint32_t)p.R};
    if (fn(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint32_t*>(w), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  // W scales: [N, K/group] bytes (a multiple of 16 per row), boxes of R rows x kSB bytes
  CUtensorMap tmS;
  {
    cuuint64_t dims[2] = {(cuuint64_t)(K / group), (cuuint64_t)N};
    cuuint64_t strides[1] = {(cuuint64_t)(K / group)};
    cuuint32_t box[2] = {(cuuint32_t)Geo<MODE>::kSB, (cuuint32_t)p.R};
    if (fn(&tmS, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(scales), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  cudaError_t e =
      cudaFuncSetAttribute(qmv_tc_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.nblk * p.split));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = (unsigned)p.split;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, qmv_tc_kernel<MODE>, tmW, tmS, x, gs_w, (int)N, (int)K, p.R, p.split,
                            p.nslots, p.wslot, p.sslot, y, d.err, inject);
}

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// Whether the tensor-core GEMV handles this NVFP4 (mode 2) or MXFP4 (mode 1)
// problem (else the mma.sync kernel does).
bool qmv_tc_supported(const DevInfo& d, int mode, int64_t N, int64_t K) {
  if (kSmemBytes > d.smem_optin || N > (int64_t)kRows * d.sm_count) return false;
  if (mode == 2) return plan_qmv_tc<2>(d, N, K).split > 0;
  if (mode == 1) return plan_qmv_tc<1>(d, N, K).split > 0;
  return false;
}

bool qmv_tc_geometry(const DevInfo& d, int64_t N, int64_t K, int* split, int* nblk, int* R, int* nslots) {
  const TcPlan p = plan_qmv_tc<2>(d, N, K);
  if (p.split == 0) return false;
  *split = p.split;
  *nblk = p.nblk;
  *R = p.R;
  *nslots = p.nslots;
  return true;
}

cudaError_t launch_qmv_tc(const DevInfo& d, int mode, const uint16_t* x, const uint32_t* w, const uint8_t* scales,
                          const float* gs_w, int64_t N, int64_t K, uint16_t* y, int inject_timeout, cudaStream_t s) {
  if (mode == 2) return launch_mode_tc<2>(d, x, w, scales, gs_w, N, K, y, inject_timeout, s);
  if (mode == 1) return launch_mode_tc<1>(d, x, w, scales, gs_w, N, K, y, inject_timeout, s);
  return cudaErrorInvalidValue;
}

}  // namespace fp4
