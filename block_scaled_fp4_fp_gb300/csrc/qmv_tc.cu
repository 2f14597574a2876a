// qmv_tc.cu -- NVFP4 / MXFP4 decode GEMV on the 5th-generation tensor cores.
//
// Pages: "epic: NVIDIA Volta (sm_70) inference acceleration program #1536"
// (Baseline: the decode step is the qmv weight stream; the V100 kernel is
// ALU-bound at 7.7 % of HBM), "mlx 0.30.7.3 -> 0.30.7.6" qqmm.cpp (the M = 1
// route: x against NVFP4 W stored [N, K]).
//
// The tensor core decodes the weights: W streams by TMA as the block-scaled
// FP4 B operand of tcgen05.mma.kind::mxf4nvf4 (E4M3 scales per 16, or E8M0
// per 32, applied by the hardware), so no instruction touches a weight.  The
// bf16 activation x is written as kTerms = 6 FP4 terms in radix 8 over one
// power-of-two scale per CTA slice of K:
//     x = 2^e0 * (sum_t d_t 2^(6 - 3t) + r),   d_t in {-4, ..., 4},
// with max|x| / 2^e0 in [128, 256).  Rounding r_t 2^(3t-6) to the nearest
// integer and subtracting keeps every digit in [-4, 4]; term t stores d_t / 2
// (0, +-0.5, ..., +-2: exact e2m1 values) under the term scale 2^(7 - 3t)
// (2^7 ... 2^-8: exact E4M3 and E8M0 values), and |r| <= 2^-10, at most 2^-17
// of max|x|.  The terms are rows 0..5 of the A operand (M = 128; rows 6..127
// feed accumulator lanes nothing reads), the W rows of the CTA are the B
// operand (N = its row count rounded up to 16, at most 256), so one MMA of
// K = 64 covers up to 256 rows: the cost of such an MMA barely depends on N.
// The MMA yields D[t, n] = sum_k d_t[k] 2^(6-3t) W[n, k] in fp32 tensor
// memory (lane t, column n); the epilogue forms y = gs_w 2^e0 sum_t D[t, n].
//
// Work split.  A cluster of `split` CTAs owns R <= 256 consecutive rows; CTA
// rank i of the cluster takes the i-th slice of the K stages (K = 256 each for
// NVFP4, 512 for MXFP4).  Each CTA sums its slice into fp32 partials; ranks
// 1.. store theirs into rank 0's shared memory with asynchronous remote stores
// (distributed shared memory) that a barrier there counts by bytes, and rank 0
// adds them in rank order -- the same order on every run -- and writes y.
//   warp 0: barrier setup (one barrier per lane), then the TMA producer: per
//           stage kCh boxes of R rows x 128 bytes of W (128-byte swizzle, so
//           rows land as the 8-row atoms the MMA reads) and one box of R rows
//           x 16 bytes of W's linear scales, into a ring sized in bytes (a
//           slot holds kCh ceil(R/8) KB of codes; up to ~200 KB, at least
//           two slots, in flight).  The first kXPre stages are issued before
//           griddepcontrol.wait (programmatic dependent launch: W is not
//           written by the kernel this one overlaps); later ones wait for the
//           x slice to land, which would otherwise queue behind them;
//   warp 1: tensor memory allocation; one thread issues each stage's 4 kCh
//           MMAs (M 128, N <= 256, K 64) into one accumulator, then one commit
//           that frees the stage's operands (and, when the ring holds fewer
//           than kMeta weight slots, a second that frees its weight slot).  B
//           rows >= R read whatever follows the slot; the accumulator columns
//           they feed are not read;
//   warps 2-17: four groups of four warps (one per tensor-memory lane
//           quadrant); group g prepares the stages i % 4 == g in operand slot
//           g: the x terms in shared memory, then, once the stage's weights
//           have landed, each warp stores the stage's W scales into the slot's
//           scale columns of its lane quadrant (tcgen05.st; B row n's scales
//           sit in lane n % 32, column (n % 128) / 32 of the k-step's group,
//           four columns further for rows 128..255).  A group that finds its
//           operand slot free again (stage i - 4 done) passes the weight slot
//           of that stage back to the TMA producer (when the ring holds kMeta
//           slots or more).  After the last stage the four warps of lane
//           quadrant 0 read D's term lanes (16x256b loads) and add them per
//           column with warp shuffles into the partials.
#include <algorithm>
#include <cstring>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace fp4 {

namespace {

constexpr int kTerms = 6;           // x expansion terms (A rows 0..5)
constexpr int kMeta = 4;            // operand slots: one per prep group
constexpr int kMaxSlots = 32;       // weight ring slots at most
constexpr uint32_t kInflightBytes = 200u * 1024u;  // weight bytes a CTA keeps in flight at most
constexpr int kXPre = 5;            // weight stages issued before x has landed (later ones wait for it)
constexpr int kChunk = 256;         // codes per TMA box (128 bytes per row)
constexpr int kRows = 256;          // W rows per CTA at most (MMA N <= 256)
constexpr int kMaxSplit = 4;        // CTAs per cluster at most (the plan takes 1, 2 or 4)
constexpr int kMaxGroup = 4;        // matrices of one grouped launch at most
constexpr int kGroups = 4;          // prep groups; group g prepares local stages i % kGroups == g
constexpr int kGroupThreads = 128;  // one group = 4 warps, one per lane quadrant
constexpr int kPrep = kGroups * kGroupThreads;
constexpr int kThreads = 64 + kPrep;  // TMA warp, MMA warp, prep warps
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfaCol = 256;   // term scales: one 4-column group
constexpr uint32_t kSfbCol = 288;   // W scales of operand slot m, k-step group j: kSfbCol + 32 m + 8 j
                                    // (rows 0..127; rows 128..255 four columns further)
static_assert(kMeta == kGroups, "group g owns operand slot g");
static_assert(kSfbCol + kMeta * 32 <= kTmemCols, "scale columns exceed the allocation");
static_assert(kMaxSlots <= 32 && kMeta <= 32, "one barrier pair per lane of warp 0");
// kind::mxf4nvf4 descriptor: E2M1 A/B, K-major, M = 128 (N is set per launch); bit 23 selects E8M0 scales
constexpr uint32_t kIdescM = (1u << 7) | (1u << 10) | ((128u >> 4) << 24);

// Per format: a stage is kCh chunks of 256 elements; a row carries kSB = 16
// scale bytes per stage, word j of which covers k-steps (K = 64) j kSpk / 4 ..
// NVFP4 (E4M3 per 16): k-step j reads word j; MXFP4 (E8M0 per 32): half j & 1
// of word j / 2, through the scale-factor id.
template <int MODE> struct Fmt;
template <> struct Fmt<2> {
  static constexpr int kCh = 1;
  static constexpr int kGroup = 16;
  static constexpr uint32_t kIdesc = kIdescM;
  // E4M3 byte of the term scale 2^(7-3t) (exact: 2^7 ... 2^-8, the last one subnormal)
  __host__ __device__ static constexpr uint32_t term_scale(int t) {
    return (7 - 3 * t >= -6) ? (uint32_t)((7 - 3 * t + 7) << 3) : (1u << (7 - 3 * t + 9));
  }
};
template <> struct Fmt<1> {
  static constexpr int kCh = 2;
  static constexpr int kGroup = 32;
  static constexpr uint32_t kIdesc = kIdescM | (1u << 23);
  // E8M0 byte of 2^(7-3t)
  __host__ __device__ static constexpr uint32_t term_scale(int t) { return (uint32_t)(127 + 7 - 3 * t); }
};
template <int MODE> struct Geo {
  static constexpr int kCh = Fmt<MODE>::kCh;
  static constexpr int kBK = 256 * kCh;               // codes per stage
  static constexpr int kSB = kBK / Fmt<MODE>::kGroup;  // scale bytes per row per stage
  static constexpr int kSpk = 64 / Fmt<MODE>::kGroup;  // scales per row per k-step
  static_assert(kSB == 16, "a row brings one 16-byte word of scales per stage");
};

// Shared memory (from a 1024-aligned base): [weight ring | term atoms |
// term-scale tile | x slice | partials | barriers].  The weight ring is split
// at launch into code slots and, after them, scale slots.
constexpr int kMaxKSlice = 17408;  // elements of x per CTA
constexpr uint32_t kSmemBytes = 227u * 1024u;
constexpr uint32_t kBarBytes = 1024;
constexpr uint32_t kRedBytes = kMaxSplit * kRows * 4;
template <int MODE> struct Lay {
  using G = Geo<MODE>;
  static constexpr uint32_t kAtoms = kMeta * G::kCh;  // term atoms: A rows 0..7 of chunk h of slot m
  static constexpr uint32_t kFixed = kAtoms * 1024 + 512 + kMaxKSlice * 2 + kRedBytes + kBarBytes + 1024;
  static constexpr uint32_t kRing = (kSmemBytes - kFixed) / 1024u * 1024u;
  static constexpr uint32_t kOffT = kRing;                     // atom kCh m + h
  static constexpr uint32_t kOffSFA = kOffT + kAtoms * 1024;  // term-scale tile
  static constexpr uint32_t kOffX = kOffSFA + 512;              // x slice (bf16)
  static constexpr uint32_t kOffRed = kOffX + kMaxKSlice * 2;  // [split][256] fp32 partials (rank 0)
  static constexpr uint32_t kOffBar = kOffRed + kRedBytes;
  static_assert(kOffBar + kBarBytes + 1024 <= kSmemBytes, "shared memory layout overflows");
  // an MMA reads 128 A rows (16 KB) from a term atom and up to 256 B rows (32 KB)
  // from a code chunk's start: both stay inside the allocation
  static_assert(kOffT + (kAtoms - 1) * 1024 + 16384 <= kOffBar, "A-operand reads past the allocation");
  static_assert(kRing + 32768 <= kOffBar, "B-operand reads past the allocation");
};
static_assert((2 * kMaxSlots + 2 * kMeta + 5) * 8 + 16 + (kPrep / 32) * 4 <= kBarBytes, "barrier area");

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

// The matrices of one launch: a plain GEMV is a group of one; a grouped GEMV
// multiplies the same x by up to kMaxGroup matrices of the same K (q, k and v
// stored apart, say).  Matrix m owns row blocks blk0[m] .. blk0[m+1]-1, its rows
// dealt out evenly over them; each has its own tensor maps, global scale and y.
struct QmvGroup {
  CUtensorMap tmW[kMaxGroup];  // codes [N_m, K/2] bytes, boxes of R rows x 128 bytes
  CUtensorMap tmS[kMaxGroup];  // linear scales [N_m, K/group], boxes of R rows x 16 bytes
  const float* gs_w[kMaxGroup];
  uint16_t* y[kMaxGroup];
  int N[kMaxGroup];
  int blk0[kMaxGroup + 1];
  int count;
};

// The GEMV launched next on the stream, if the caller names it: once all of a
// CTA's own weights have landed, its producer warms L2 with the first `stages`
// weight boxes the same-numbered CTAs of that launch will read (TMA tensor
// prefetches through that launch's own maps), so that DRAM keeps streaming
// while this launch finishes, and the next launch's first stages -- and the x
// loads that queue behind them -- come from L2.  A hint only: nothing is written.
struct QmvNext {
  CUtensorMap tmW[kMaxGroup];
  CUtensorMap tmS[kMaxGroup];
  int N[kMaxGroup];
  int blk0[kMaxGroup + 1];
  int count = 0;  // 0: no prefetch
  int split = 1, K = 0, stages = 0;
};

template <int MODE, bool QX>
__global__ void __launch_bounds__(kThreads, 1) qmv_tc_kernel(const __grid_constant__ QmvGroup mats,
                                                              const __grid_constant__ QmvNext next,
                                                              const uint16_t* __restrict__ x,
                                                              const float* __restrict__ gs_x, int K,
                                                              int R, int split, int nslots, uint32_t wslot,
                                                              uint32_t sslot, unsigned* __restrict__ err,
                                                              int inject_timeout) {
  using F = Fmt<MODE>;
  using G = Geo<MODE>;
  using L = Lay<MODE>;
  constexpr int kCh = G::kCh;
  constexpr int kBK = G::kBK;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  uint64_t* wfull = reinterpret_cast<uint64_t*>(smem + L::kOffBar);  // weight slot landed (TMA bytes)
  uint64_t* wempty = wfull + kMaxSlots;                           // weight slot consumed (relayed)
  uint64_t* mfull = wempty + kMaxSlots;                           // stage operands built (prep group)
  uint64_t* mempty = mfull + kMeta;                               // stage operands consumed (MMA commit)
  uint64_t* done = mempty + kMeta;
  uint64_t* pbar = done + 1;  // rank 0: the other ranks' partials have landed (byte count)
  uint64_t* tbar = pbar + 1;  // warp 1 has allocated tensor memory (tmem_slot written)
  uint64_t* never = tbar + 1; // fault injection: a barrier nothing arrives at
  uint64_t* xin = never + 1;   // the x slice has landed in shared memory (one arrival)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(xin + 1);
  uint32_t* red = tmem_slot + 4;  // kPrep / 32 warp maxima of |x| (bf16 bits)
  float* part = reinterpret_cast<float*>(smem + L::kOffRed);
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem + L::kOffX);
  const uint32_t offS = (uint32_t)nslots * wslot;  // linear-scale slots follow the code slots
  const uint32_t wchunk = wslot / kCh;              // one 256-element chunk of a code slot

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = (int)(blockIdx.x % (unsigned)split);  // rank within the cluster (clusters are consecutive)
  const int blk = (int)(blockIdx.x / (unsigned)split);
  int mi = 0;  // this CTA's matrix
  while (mi + 1 < mats.count && blk >= mats.blk0[mi + 1]) ++mi;
  const int lb = blk - mats.blk0[mi], nblk = mats.blk0[mi + 1] - mats.blk0[mi];
  const int r0 = (int)(((int64_t)mats.N[mi] * lb) / nblk);
  const int r1 = (int)(((int64_t)mats.N[mi] * (lb + 1)) / nblk);
  const CUtensorMap* tmW = &mats.tmW[mi];
  const CUtensorMap* tmS = &mats.tmS[mi];
  const int rows = r1 - r0;  // <= R <= 256
  const int nmma = (R + 15) & ~15;  // MMA N
  const int nkb = K / kBK;
  const int kb0 = (int)(((int64_t)nkb * rank) / split);
  const int nst = (int)(((int64_t)nkb * (rank + 1)) / split) - kb0;  // this CTA's stages (>= 1)
  // weight slots go back to the TMA producer through the prep group that reuses the
  // stage's operand slot (kMeta stages later), or, when the ring holds fewer than
  // kMeta slots, through a second MMA commit per stage
  const bool relay = nslots >= kMeta;

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
      mbar_init(pbar, 1);
      mbar_init(tbar, 1);
      mbar_init(never, 1);
      mbar_init(xin, 1);
    }
    fence_barrier_init();  // release of the barrier inits to the cluster
  }
  // Ranks > 0 wait on this arrival before storing into rank 0's shared memory:
  // rank 0 has started and its barriers are initialized.
  __syncwarp();
  if (split > 1) cluster_arrive_relaxed();
  // The constant term-scale tile (A scales): row t < 6 holds the weight
  // 2^(7-3t) of term t for each of the k-step's four blocks; the other rows
  // are zero.  tcgen05.cp gives lane t (quadrant 0) these bytes in its column.
  if (threadIdx.x < 128) {
    const int row = threadIdx.x >> 2, word = threadIdx.x & 3;
    const uint32_t v = (row < kTerms && word == 0) ? F::term_scale(row) * 0x01010101u : 0u;
    reinterpret_cast<uint32_t*>(smem + L::kOffSFA)[threadIdx.x] = v;
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncthreads();
  bool failed = false;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer (weights)
    if (elect_one_sync()) {
      prefetch_tmap(tmW);
      prefetch_tmap(tmS);
      // out-of-range rows are zero-filled and counted
      const uint32_t tx = (uint32_t)R * (128u * kCh + G::kSB);
      int s = 0, round = 0;
      for (int i = 0; i < nst; ++i) {
        // The x loads are issued after griddepcontrol.wait and queue behind this SM's
        // weight requests: past the first kXPre stages the stream waits for x to land
        // (measured +0.6 % on the fused decode stack).
        if (i == kXPre) mbar_wait(xin, 0, err, failed);
        if (round > 0) mbar_wait(&wempty[s], (round - 1) & 1, err, failed);
        mbar_arrive_expect_tx(&wfull[s], tx);
#pragma unroll
        for (int h = 0; h < kCh; ++h)
          tma_load_2d(smem + s * wslot + h * wchunk, tmW, &wfull[s], ((kb0 + i) * kCh + h) * 128, r0);
        tma_load_2d(smem + offS + s * sslot, tmS, &wfull[s], (kb0 + i) * G::kSB, r0);
        if (++s == nslots) { s = 0; ++round; }
      }
      // no copy may still be writing shared memory when the CTA exits (the waits
      // run, bounded, even after an earlier one expired)
      bool drain_failed = false;
      for (int i = max(0, nst - nslots); i < nst; ++i)
        mbar_wait(&wfull[i % nslots], (i / nslots) & 1, err, drain_failed);
      // every weight byte of this CTA has landed: warm L2 for the next launch (see
      // QmvNext).  Issued any earlier, the prefetches compete with the last CTAs'
      // own loads and lengthen this launch (measured on the fused decode stack).
      if (next.count > 0) {
        const int ncta = next.blk0[next.count] * next.split;
        const int nkb = next.K / kBK;
        for (int c = blockIdx.x; c < ncta; c += gridDim.x) {
          const int nrank = c % next.split, nb = c / next.split;
          int m = 0;
          while (m + 1 < next.count && nb >= next.blk0[m + 1]) ++m;
          const int lb = nb - next.blk0[m], cnt = next.blk0[m + 1] - next.blk0[m];
          const int nr0 = (int)(((int64_t)next.N[m] * lb) / cnt);
          const int k0 = (int)(((int64_t)nkb * nrank) / next.split);
          const int k1 = min((int)(((int64_t)nkb * (nrank + 1)) / next.split), k0 + next.stages);
          for (int kb = k0; kb < k1; ++kb) {
#pragma unroll
            for (int h = 0; h < kCh; ++h)
              asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];"
                           :: "l"(&next.tmW[m]), "r"((kb * kCh + h) * 128), "r"(nr0) : "memory");
            asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];"
                         :: "l"(&next.tmS[m]), "r"(kb * G::kSB), "r"(nr0) : "memory");
          }
        }
      }
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
    const uint32_t tmem = *tmem_slot;
    if (lane == 0) mbar_arrive(tbar);  // releases the tmem_slot write to the prep warps
    if (elect_one_sync()) {
      if (inject_timeout) {
        bool injected = false;  // separate flag: the injected expiry must not stop later waits
        mbar_wait(never, 0, err, injected, 2000000LL);
      }
      asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;"
                   :: "r"(tmem + kSfaCol), "l"(desc_sf(base + L::kOffSFA)) : "memory");
      const uint32_t idesc_n = F::kIdesc | ((uint32_t)(nmma >> 3) << 17);
      int m = 0, s = 0;
      for (int i = 0; i < nst; ++i) {
        mbar_wait(&mfull[m], (i / kMeta) & 1, err, failed);  // the group also saw the weights land
        tc_fence_after();
        const uint32_t sfb_t = tmem + kSfbCol + 32 * m;  // 4-column aligned groups
#pragma unroll
        for (int j = 0; j < 4 * kCh; ++j) {
          // k-step j (K = 64): chunk h = j / 4, 32 bytes further per k-step along the swizzled rows
          const int h = j >> 2, jj = j & 3;
          // A: the chunk's term atom (rows 8..127 read the atoms after it); B: the W rows
          const uint64_t adesc = desc_sw128(base + L::kOffT + (m * kCh + h) * 1024, 1024) + (uint64_t)(2 * jj);
          const uint64_t bdesc = desc_sw128(base + s * wslot + h * wchunk, 1024) + (uint64_t)(2 * jj);
          // scale words: group (j kSpk) / 4, scale-factor id (j kSpk) % 4
          const uint32_t grp = (uint32_t)((j * G::kSpk) >> 2);
          const uint32_t sf_id = (uint32_t)((j * G::kSpk) & 3);
          const uint32_t idesc = idesc_n | (sf_id << 29) | (sf_id << 4);
          const uint32_t acc = (i > 0 || j > 0) ? 1u : 0u;
          if (MODE == 2)
            asm volatile(
                "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %6, 0;\n\t"
                "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
                :: "r"(tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(tmem + kSfaCol), "r"(sfb_t + 8 * grp),
                   "r"(acc) : "memory");
          else
            asm volatile(
                "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %6, 0;\n\t"
                "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
                :: "r"(tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(tmem + kSfaCol), "r"(sfb_t + 8 * grp),
                   "r"(acc) : "memory");
        }
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                     :: "r"(smem_u32(&mempty[m])) : "memory");
        if (!relay)
          asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                       :: "r"(smem_u32(&wempty[s])) : "memory");
        if (++m == kMeta) m = 0;
        if (++s == nslots) s = 0;
      }
      asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                   :: "r"(smem_u32(done)) : "memory");
    }
  } else {
    // ------------------------------------------- prep warps (2..17), then epilogue
    const int pa = threadIdx.x - 64;           // 0..kPrep-1
    const int grp = pa / kGroupThreads;        // prep group = operand slot
    const int pt = pa % kGroupThreads;         // thread within the group
    if (split > 1 && rank > 0) cluster_wait();  // (see the arrival after the barrier inits)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // this CTA's slice of x (bf16, nst * kBK * 2 bytes) -> shared memory and its max|x|,
    // by ordinary loads: a bulk copy would queue behind the weight boxes already in
    // flight from this SM
    const uint4* xg = reinterpret_cast<const uint4*>(x + (int64_t)kb0 * kBK);
    const int nx = nst * (kBK / 8);  // 16-byte chunks of the slice
    constexpr int kXLoads = (kMaxKSlice / 8 + kPrep - 1) / kPrep;
    uint4 xq[kXLoads];
#pragma unroll
    for (int u = 0; u < kXLoads; ++u)  // every load in flight before the first use
      xq[u] = pa + kPrep * u < nx ? __ldg(xg + pa + kPrep * u) : make_uint4(0, 0, 0, 0);
    if (QX) {
      // The quantized-activation route: x is replaced by fp_dequantize(fp_quantize(x))
      // (bf16) before the GEMV.  A block (16 or 32 elements) is the 16-byte pieces of
      // 2 or 4 neighbouring lanes (the slice starts on a block boundary); the slice is
      // a multiple of 32 pieces, so the range test is uniform across each warp.
      const float gsx = (MODE == 2 && gs_x) ? __ldg(gs_x) : 1.0f;
#pragma unroll
      for (int u = 0; u < kXLoads; ++u) {
        if (pa + kPrep * u >= nx) break;
        uint32_t mb = max_mag8(xq[u]);
        mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
        if (MODE == 1) mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
        float mul, sval;
        uint32_t sbyte;
        block_scale_rule<MODE>(mb, gsx, mul, sbyte, sval);
        xq[u] = quant_dequant8(xq[u], mul, sval, gsx);
      }
    }
    uint32_t m2 = 0;
#pragma unroll
    for (int u = 0; u < kXLoads; ++u) {
      if (pa + kPrep * u < nx) reinterpret_cast<uint4*>(xs)[pa + kPrep * u] = xq[u];
      m2 = __vmaxu2(m2, xq[u].x & 0x7FFF7FFFu);
      m2 = __vmaxu2(m2, xq[u].y & 0x7FFF7FFFu);
      m2 = __vmaxu2(m2, xq[u].z & 0x7FFF7FFFu);
      m2 = __vmaxu2(m2, xq[u].w & 0x7FFF7FFFu);
    }
    const uint32_t mb = __reduce_max_sync(0xffffffffu, max(m2 & 0xFFFFu, m2 >> 16));
    if (lane == 0) red[pa >> 5] = mb;
    asm volatile("bar.sync 1, %0;" :: "n"(kPrep) : "memory");  // prep warps only; x is in shared memory
    if (pa == 0) mbar_arrive(xin);
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
    const uint32_t tmem = *tmem_slot;
    const int q4 = warp & 3;
    const uint32_t sfb_lane = tmem + ((uint32_t)(32 * q4) << 16) + kSfbCol + 32 * grp;
    // stage bookkeeping: weight slot s (round wr) of stage i (the ring may hold
    // fewer slots than there are groups)
    int s = grp % nslots, wr = grp / nslots;
    const int lo = pt & 15, hi4 = ((pt >> 4) & 7) << 4;
    for (int i = grp; i < nst; i += kGroups) {
      if (i >= kMeta) {
        mbar_wait(&mempty[grp], ((i / kMeta) - 1) & 1, err, failed);  // stage i - kMeta is done
        tc_fence_after();  // its MMAs have read the slot's terms and scale columns
        if (relay && pt == 0) {
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
        uint8_t* tatom = smem + L::kOffT + (grp * kCh + h) * 1024;
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
          // byte pt of A row t, 128-byte swizzle
          tatom[t * 128 + ((hi4 ^ (t << 4))) + lo] = code;
        }
      }
      // (b) the stage's W scales, once it has landed.  B row n's scale word j sits in
      // lane n % 32 (written in every lane quadrant), column 8j + n / 32 for rows
      // 0..127 and 8j + 4 + (n - 128) / 32 for rows 128..255; this thread moves
      // rows 32c + lane (c = 0..7).  Rows >= rows get 0.
      if (!relay && i >= nslots) {
        // the slot's previous stage (i - nslots) is done with it, so the producer has
        // (or will have) issued this stage's load and wfull[s] is at most one phase
        // behind the phase waited for below
        const int ip = i - nslots;
        mbar_wait(&mempty[ip % kMeta], (ip / kMeta) & 1, err, failed);
      }
      mbar_wait(&wfull[s], wr & 1, err, failed);
      const uint8_t* sc = smem + offS + s * sslot;
      if (nmma > 128) {  // warp-uniform
        uint4 v[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const int row = 32 * c + lane;
          v[c] = row < rows ? *reinterpret_cast<const uint4*>(sc + row * G::kSB) : make_uint4(0, 0, 0, 0);
        }
        asm volatile(
            "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
            "%13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
            :: "r"(sfb_lane), "r"(v[0].x), "r"(v[1].x), "r"(v[2].x), "r"(v[3].x), "r"(v[4].x), "r"(v[5].x), "r"(v[6].x),
               "r"(v[7].x), "r"(v[0].y), "r"(v[1].y), "r"(v[2].y), "r"(v[3].y), "r"(v[4].y), "r"(v[5].y), "r"(v[6].y),
               "r"(v[7].y), "r"(v[0].z), "r"(v[1].z), "r"(v[2].z), "r"(v[3].z), "r"(v[4].z), "r"(v[5].z), "r"(v[6].z),
               "r"(v[7].z), "r"(v[0].w), "r"(v[1].w), "r"(v[2].w), "r"(v[3].w), "r"(v[4].w), "r"(v[5].w), "r"(v[6].w),
               "r"(v[7].w) : "memory");
      } else {  // N <= 128: the MMA reads only the first four columns of each group
        uint4 v[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int row = 32 * c + lane;
          v[c] = row < rows ? *reinterpret_cast<const uint4*>(sc + row * G::kSB) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t* w = reinterpret_cast<const uint32_t*>(v);  // word j of row c at w[4 c + j]
          asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};"
                       :: "r"(sfb_lane + 8 * j), "r"(w[j]), "r"(w[4 + j]), "r"(w[8 + j]), "r"(w[12 + j]) : "memory");
        }
      }
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      tc_fence_before();
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the term bytes, for the MMA
      mbar_arrive(&mfull[grp]);
      s += kGroups;
      while (s >= nslots) { s -= nslots; ++wr; }
    }
    // ---- epilogue: the lane-quadrant-0 warps (one per group) each take 64
    // columns of D.  A 16x256b load gives thread T lane T / 4 (and lane T / 4 + 8)
    // at columns 8 j + 2 (T % 4) + {0, 1} of each 8-column block j; the sum over
    // the term lanes 0..5 is a butterfly over T's bits 2..4, after which thread T
    // keeps block T / 4.  partial = 2^e0 sum_t D[t, n].
    if (q4 == 0) {
      mbar_wait(done, 0, err, failed);
      tc_fence_after();
      const int c0 = 64 * grp;
      float sum[2] = {0.f, 0.f};
      if (c0 < nmma) {  // warp-uniform
        uint32_t d[2][16];
#pragma unroll
        for (int h = 0; h < 2; ++h)
          asm volatile(
              "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
              : "=r"(d[h][0]), "=r"(d[h][1]), "=r"(d[h][2]), "=r"(d[h][3]), "=r"(d[h][4]), "=r"(d[h][5]),
                "=r"(d[h][6]), "=r"(d[h][7]), "=r"(d[h][8]), "=r"(d[h][9]), "=r"(d[h][10]), "=r"(d[h][11]),
                "=r"(d[h][12]), "=r"(d[h][13]), "=r"(d[h][14]), "=r"(d[h][15])
              : "r"(tmem + (uint32_t)(c0 + 32 * h)));
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        const bool term = (lane >> 2) < kTerms;
#pragma unroll
        for (int b = 0; b < 8; ++b) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            float v = term ? __uint_as_float(d[b >> 2][4 * (b & 3) + e]) : 0.f;
            v += __shfl_xor_sync(0xffffffffu, v, 4);
            v += __shfl_xor_sync(0xffffffffu, v, 8);
            v += __shfl_xor_sync(0xffffffffu, v, 16);
            if (b == (lane >> 2)) sum[e] = v;
          }
        }
      }
      const int nb = c0 + 8 * (lane >> 2) + 2 * (lane & 3);  // this thread's columns nb, nb + 1
      float partial[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) partial[k] = finite ? ldexpf(sum[k], e0) : __int_as_float(0x7FC00000);
      if (rank > 0) {
        // asynchronous stores into rank 0's partials; its barrier counts the bytes
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int n = nb + k;
          if (n < rows)
            asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];"
                         :: "r"(map_rank(part + rank * kRows + n, 0)), "r"(__float_as_uint(partial[k])),
                            "r"(map_rank(pbar, 0)) : "memory");
        }
      } else {
        if (split > 1) {
          if (grp == 0 && lane == 0) mbar_arrive_expect_tx(pbar, (uint32_t)(split - 1) * (uint32_t)rows * 4u);
          mbar_wait(pbar, 0, err, failed);  // every other rank's partials have landed
        }
        const float g = mats.gs_w[mi] ? __ldg(mats.gs_w[mi]) : 1.0f;
        uint16_t* y = mats.y[mi];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int n = nb + k;
          if (n < rows) {
            float acc_y = partial[k];
            for (int c = 1; c < split; ++c) acc_y += part[c * kRows + n];
            y[r0 + n] = (uint16_t)f32_to_bf16_rn(acc_y * g);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(*tmem_slot), "r"(kTmemCols) : "memory");
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
  if (cudaFuncSetAttribute(qmv_tc_kernel<MODE, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) ==
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
    if (cudaOccupancyMaxActiveClusters(&n, qmv_tc_kernel<MODE, false>, &cfg) != cudaSuccess) {
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

// The weight ring for blocks of at most R rows: slot sizes, and up to ~200 KB in
// flight (about the whole ring: measured +1.3 % over 128 KB on the fused decode
// stack, whose launches start with the ring filling while x is read), at least
// kMeta slots if it can (for the slot relay) and at least two.  False if two
// slots do not fit.
template <int MODE>
bool size_ring(TcPlan& p, int R) {
  using G = Geo<MODE>;
  p.R = R;
  p.wslot = (uint32_t)G::kCh * (uint32_t)((R + 7) / 8) * 1024u;
  p.sslot = ((uint32_t)R * G::kSB + 127u) / 128u * 128u;
  const uint32_t slot = p.wslot + p.sslot;
  if (Lay<MODE>::kRing / slot < 2u) return false;
  p.nslots = (int)std::min<uint32_t>(kMaxSlots, Lay<MODE>::kRing / slot);
  p.nslots = std::max<int>(std::min<int>(p.nslots, kMeta), std::min<int>(p.nslots, kInflightBytes / slot));
  return true;
}

// Choose the row blocks and the K split (1, 2 or 4 CTAs per cluster: clusters
// of 3, 5 or more measured slower to schedule).  A CTA's time is about the
// larger of its MMA issue time (stages x about 0.2 us per 4 MMAs of K = 64,
// whatever N) and its bytes at an even share of HBM bandwidth among the CTAs
// (capped at what one SM draws), plus a small cost per stage and a fixed cost
// for a cluster launch and the partial exchange; the plan with the smallest
// estimate wins (ties go to the smaller split).  The weight ring holds about
// 200 KB in flight, at least kMeta slots if it can (for the slot relay) and
// at least two.
template <int MODE>
TcPlan plan_qmv_tc(const DevInfo& d, int64_t N, int64_t K) {
  using G = Geo<MODE>;
  constexpr int kCh = G::kCh;
  constexpr int kBK = G::kBK;
  TcPlan best;
  if (K % kBK != 0 || N < 1 || d.sm_count < 1) return best;
  const int64_t nkb = K / kBK;
  const double stage_us = 0.2 * kCh, hbm_gbs = 6500.0, sm_gbs = 80.0, per_stage_us = 0.05, cluster_us = 0.6;
  double best_cost = 0.0;
  for (int split : {1, 2, 4}) {
    if (nkb < split) break;
    const int64_t nst = (nkb + split - 1) / split;
    if (nst * kBK > kMaxKSlice) continue;
    int64_t nblk = split == 1 ? d.sm_count : std::min<int64_t>(max_clusters<MODE>(d, split), d.sm_count / split);
    nblk = std::min<int64_t>(nblk, N);
    if (nblk < 1) continue;
    const int64_t R = (N + nblk - 1) / nblk;
    if (R > kRows) continue;
    const uint32_t wslot = (uint32_t)kCh * (uint32_t)((R + 7) / 8) * 1024u;
    const uint32_t sslot = ((uint32_t)R * G::kSB + 127u) / 128u * 128u;
    if (Lay<MODE>::kRing / (wslot + sslot) < 2u) continue;
    const double bw = std::min(sm_gbs, hbm_gbs / (double)(nblk * split));
    const double bytes = (double)nst * (double)R * (128.0 * kCh + G::kSB);
    const double cost = std::max((double)nst * stage_us, bytes / (bw * 1e3)) + (double)nst * per_stage_us +
                        (split > 1 ? cluster_us : 0.0);
    if (best.split == 0 || cost < best_cost) {
      best_cost = cost;
      best.split = split;
      best.nblk = (int)nblk;
      best.R = (int)R;
      best.wslot = wslot;
      best.sslot = sslot;
    }
  }
  if (best.split == 0) return best;
  size_ring<MODE>(best, best.R);
  return best;
}

// The plan of a group: the single-matrix plan of all its rows stacked (split,
// number of row blocks); for more than one matrix, the smallest block height R
// that deals every matrix whole blocks within that number of blocks.
template <int MODE>
TcPlan plan_group_tc(const DevInfo& d, int count, const int64_t* N, int64_t K, int* nb) {
  int64_t total = 0;
  for (int i = 0; i < count; ++i) total += N[i];
  TcPlan p = plan_qmv_tc<MODE>(d, total, K);
  if (p.split == 0) return p;
  if (count == 1) {
    nb[0] = p.nblk;
    return p;
  }
  for (int R = (int)((total + p.nblk - 1) / p.nblk); R <= kRows; ++R) {
    int64_t blocks = 0;
    for (int i = 0; i < count; ++i) blocks += (N[i] + R - 1) / R;
    if (blocks <= p.nblk) {
      if (!size_ring<MODE>(p, R)) break;
      for (int i = 0; i < count; ++i) nb[i] = (int)((N[i] + R - 1) / R);
      return p;
    }
  }
  p.split = 0;
  return p;
}

// The tensor maps of one matrix for blocks of R rows: codes [N, K/2] bytes in
// boxes of R rows x 128 bytes (128-byte swizzle), scales [N, K/group] bytes (a
// multiple of 16 per row) in boxes of R rows x 16 bytes.
template <int MODE>
bool encode_maps(CUtensorMap* tmW, CUtensorMap* tmS, const uint32_t* w, const uint8_t* scales, int64_t N, int64_t K,
                 int R) {
  auto fn = encode_fn();
  if (!fn) return false;
  const int group = MODE == 2 ? 16 : 32;
  cuuint32_t estr[2] = {1, 1};
  cuuint64_t dims[2] = {(cuuint64_t)(K / 2), (cuuint64_t)N};
  cuuint64_t strides[1] = {(cuuint64_t)(K / 2)};
  cuuint32_t box[2] = {128, (cuuint32_t)R};
  if (fn(tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint32_t*>(w), dims, strides, box, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  cuuint64_t sdims[2] = {(cuuint64_t)(K / group), (cuuint64_t)N};
  cuuint64_t sstrides[1] = {(cuuint64_t)(K / group)};
  cuuint32_t sbox[2] = {(cuuint32_t)Geo<MODE>::kSB, (cuuint32_t)R};
  return fn(tmS, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(scales), sdims, sstrides, sbox, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// stages of the next launch's CTAs warmed in L2: measured on the fused decode
// stack, 1-4 after this CTA's loads land give +2.5 points of HBM (NVFP4) and
// +2-4 (MXFP4), 3 the best for both; 6 or 12 lose
constexpr int kPrefetchStages = 3;

template <int MODE, bool QX>
cudaError_t launch_group_tc(const DevInfo& d, const uint16_t* x, const float* gs_x, int count,
                            const uint32_t* const* w, const uint8_t* const* scales, const float* const* gs_w,
                            const int64_t* N, int64_t K, uint16_t* const* y, const GemvGroupDesc* nextd, int inject,
                            cudaStream_t s) {
  if (count < 1 || count > kMaxGroup) return cudaErrorInvalidValue;
  int nb[kMaxGroup] = {0, 0, 0, 0};
  const TcPlan p = plan_group_tc<MODE>(d, count, N, K, nb);
  if (p.split == 0) return cudaErrorInvalidValue;
  QmvGroup g;
  memset(&g, 0, sizeof(g));
  g.count = count;
  for (int i = 0; i < count; ++i) {
    if (!encode_maps<MODE>(&g.tmW[i], &g.tmS[i], w[i], scales[i], N[i], K, p.R)) return cudaErrorInvalidValue;
    g.gs_w[i] = gs_w ? gs_w[i] : nullptr;
    g.y[i] = y[i];
    g.N[i] = (int)N[i];
    g.blk0[i + 1] = g.blk0[i] + nb[i];
  }
  // the next launch's plan, as that launch will make it (a hint: dropped if it has none)
  QmvNext nx;
  memset(&nx, 0, sizeof(nx));
  if (nextd && nextd->count >= 1 && nextd->count <= kMaxGroup) {
    int nnb[kMaxGroup] = {0, 0, 0, 0};
    const TcPlan np = plan_group_tc<MODE>(d, nextd->count, nextd->N, nextd->K, nnb);
    bool ok = np.split > 0;
    for (int i = 0; ok && i < nextd->count; ++i) {
      ok = encode_maps<MODE>(&nx.tmW[i], &nx.tmS[i], nextd->w[i], nextd->scales[i], nextd->N[i], nextd->K, np.R);
      nx.N[i] = (int)nextd->N[i];
      nx.blk0[i + 1] = nx.blk0[i] + nnb[i];
    }
    if (ok) {
      nx.count = nextd->count;
      nx.split = np.split;
      nx.K = (int)nextd->K;
      nx.stages = kPrefetchStages;
    } else {
      memset(&nx, 0, sizeof(nx));
    }
  }
  cudaError_t e =
      cudaFuncSetAttribute(qmv_tc_kernel<MODE, QX>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(g.blk0[count] * p.split));
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
  return cudaLaunchKernelEx(&cfg, qmv_tc_kernel<MODE, QX>, g, nx, x, gs_x, (int)K, p.R, p.split, p.nslots, p.wslot,
                            p.sslot, d.err, inject);
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
  return qmv_tc_group_supported(d, mode, 1, &N, K);
}

bool qmv_tc_group_supported(const DevInfo& d, int mode, int count, const int64_t* N, int64_t K) {
  if (count < 1 || count > kMaxGroup || kSmemBytes > d.smem_optin) return false;
  int64_t total = 0;
  for (int i = 0; i < count; ++i) total += N[i];
  if (total > (int64_t)kRows * d.sm_count) return false;
  int nb[kMaxGroup];
  if (mode == 2) return plan_group_tc<2>(d, count, N, K, nb).split > 0;
  if (mode == 1) return plan_group_tc<1>(d, count, N, K, nb).split > 0;
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

cudaError_t launch_qmv_tc_group(const DevInfo& d, int mode, const uint16_t* x, const float* gs_x, int qx, int count,
                                const uint32_t* const* w, const uint8_t* const* scales, const float* const* gs_w,
                                const int64_t* N, int64_t K, uint16_t* const* y, const GemvGroupDesc* next,
                                int inject_timeout, cudaStream_t s) {
  if (mode == 2 && qx)
    return launch_group_tc<2, true>(d, x, gs_x, count, w, scales, gs_w, N, K, y, next, inject_timeout, s);
  if (mode == 1 && qx)
    return launch_group_tc<1, true>(d, x, gs_x, count, w, scales, gs_w, N, K, y, next, inject_timeout, s);
  if (mode == 2)
    return launch_group_tc<2, false>(d, x, nullptr, count, w, scales, gs_w, N, K, y, next, inject_timeout, s);
  if (mode == 1)
    return launch_group_tc<1, false>(d, x, nullptr, count, w, scales, gs_w, N, K, y, next, inject_timeout, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_qmv_tc(const DevInfo& d, int mode, const uint16_t* x, const float* gs_x, int qx,
                          const uint32_t* w, const uint8_t* scales, const float* gs_w, int64_t N, int64_t K,
                          uint16_t* y, int inject_timeout, cudaStream_t s) {
  return launch_qmv_tc_group(d, mode, x, gs_x, qx, 1, &w, &scales, &gs_w, &N, K, &y, nullptr, inject_timeout, s);
}

}  // namespace fp4
