// qmv_affine.cu -- affine 4-bit decode GEMV (group 32 / 64 / 128, bf16 scale
// and bias) on the 5th-generation tensor cores.
//
// Pages: "epic: NVIDIA Volta (sm_70) inference acceleration program #1536"
// (Baseline: the decode step streams affine 4-bit group-64 weights at 7.7 % of
// the V100's bandwidth, ALU-bound; Diagnosis 3: the accumulator type -- fp32
// here), "mlx 0.30.7.3 -> 0.30.7.6" quantized.cpp (affine w = q * scale + bias).
//
// y[n] = sum_g s[n,g] (sum_{k in g} q[n,k] x[k]) + b[n,g] X_g, X_g = sum_{k in g} x[k].
// The weight stream is the cost, so per weight the kernel spends well under
// one instruction, and the tensor core keeps every scale group apart:
//   * warp 16 streams W by TMA, one box of R rows x 128 bytes (256 codes,
//     128-byte swizzle) per stage, and per window of 16 scale groups one box of
//     R rows of scales and one of biases.  Stages issued before the previous
//     kernel ends (programmatic dependent launch) read only W, which no kernel of
//     this library writes and releases early;
//   * warps 0-15 decode: row r of the CTA lives in tensor-memory lane
//     32 (r % 4) + r / 4; warp w (lane quadrant w % 4) takes 64 codes of each
//     of its rows per stage.  One LOP3 turns a code pair into an f16 pair --
//     (w & 0x000F000F) | 0x64006400 is f16(1024 + q) for nibbles 0 and 4,
//     (w & 0x00F000F0) | 0x64006400 is f16(1024 + 16 q) for nibbles 1 and 5,
//     the same on w >> 8 for nibbles 2, 6 and 3, 7 -- and tcgen05.st writes the
//     pairs into the stage's A operand in tensor memory (M = 128 rows, K along
//     columns).  The same warps write the stage's B operand into shared memory:
//     N = 16 columns, column j holding x (pre-scaled f16, in the A operand's k
//     order, divided by 16 where A carries 16 q) over the k-steps of scale group
//     j of the current window and zeros elsewhere;
//   * warp 17 issues tcgen05.mma.kind::f16 (A from tensor memory, B from shared
//     memory, M 128, N 16, K 16): D[n, j] = sum over group j of (1024 + c q) x / c
//     = 1024 X'_j + (sum q x)_j, each group in its own fp32 column;
//   * warps 18-21 drain each window's D (double-buffered) and accumulate
//     y[n] += 2^-sigma_j (s (D - 1024 X'_j) + b X_j) in fp32 (sigma_j: the group's
//     power-of-two pre-scale of x, max|x| 2^sigma in [2^14, 2^15), exact in f16
//     down to 2^-24 of the group's max).
// Every mbarrier wait is bounded (an expired wait records FP4_ERR_TIMEOUT).
#include <algorithm>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "launch.h"

namespace fp4 {

namespace {

constexpr int kDecWarps = 16;
constexpr int kProdWarp = 16, kMmaWarp = 17;  // warps 18-21: epilogue (one per lane quadrant)
constexpr int kThreads = 22 * 32;
constexpr int kRows = 128;            // rows per CTA at most (one MMA of M = 128)
constexpr int kStageCodes = 256;      // codes per row per stage (one 128-byte TMA box)
constexpr int kWinGroups = 16;        // scale groups per window (the MMA's N)
constexpr int kMaxK = 32768;
constexpr int kOpSlots = 2;           // A (tensor memory) and B (shared memory) operand slots
constexpr int kScaleSlots = 3;
constexpr int kMaxCodeSlots = 16;
constexpr uint32_t kBStage = 8192;    // B operand of a stage: 4 blocks of 16 rows x 128 bytes
constexpr uint32_t kScaleSlot = 2u * kRows * 32u;  // scales then biases, 32 bytes per row
constexpr uint32_t kSmemBytes = 227u * 1024u;
constexpr uint32_t kBarBytes = 512;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAcol = 0;         // A slot s at columns 128 s
constexpr uint32_t kDcol = 256;       // D buffer d at columns 256 + 32 d
// kind::f16 descriptor: fp32 accumulator, f16 A and B, both K-major, N = 16, M = 128
constexpr uint32_t kIdesc = (1u << 4) | ((16u >> 3) << 17) | ((128u >> 4) << 24);
static_assert(2 * kMaxCodeSlots + 2 * kOpSlots + 2 * kScaleSlots + 4 + 1 <= kBarBytes / 8, "barrier area");

__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}

__device__ __forceinline__ uint32_t f16x2_bits(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               :: "r"(smem_u32(bar)) : "memory");
}

struct AffGeo {
  int nblk = 0;        // CTAs (row blocks)
  int R = 0;           // rows per CTA at most (blocks own R or R - 1)
  int ncs = 0;         // code ring slots
  uint32_t cslot = 0;  // bytes per code slot (ceil(R / 8) swizzle atoms)
};

// Shared memory (from a 1024-aligned base):
// [code ring | B slots | scale slots | x16 (K f16) | group arrays (3 x K/group floats) | barriers]
__host__ __device__ inline uint32_t fixed_bytes(int K, int group) {
  return (uint32_t)kOpSlots * kBStage + (uint32_t)kScaleSlots * kScaleSlot + (uint32_t)K * 2u +
         3u * 4u * (uint32_t)(K / group) + kBarBytes;
}

template <int GROUP>
__global__ void __launch_bounds__(kThreads, 1) qmv_affine_kernel(
    const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmS,
    const __grid_constant__ CUtensorMap tmB, const uint16_t* __restrict__ x, int N, int K, AffGeo geo,
    uint16_t* __restrict__ y, unsigned* __restrict__ err) {
  constexpr int kLpg = GROUP / 8;                      // 16-byte x pieces per group
  constexpr int kSpw = kWinGroups * GROUP / kStageCodes;  // stages per full window
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t ring = (uint32_t)geo.ncs * geo.cslot;
  const uint32_t offB = ring;
  const uint32_t offS = offB + kOpSlots * kBStage;
  const uint32_t offX = offS + kScaleSlots * kScaleSlot;
  const int ngroups = K / GROUP;
  uint16_t* x16 = reinterpret_cast<uint16_t*>(smem + offX);          // pre-scaled x in the A operand's k order
  float* ginv = reinterpret_cast<float*>(smem + offX + (uint32_t)K * 2u);  // 2^-sigma of group g
  float* gx1 = ginv + ngroups;                                        // X'_g: sum of the staged values
  float* gx2 = gx1 + ngroups;                                         // X_g: sum of pre-scaled x
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + offX + (uint32_t)K * 2u + 12u * (uint32_t)ngroups);
  uint64_t* cfull = bars;
  uint64_t* cempty = cfull + kMaxCodeSlots;
  uint64_t* ofull = cempty + kMaxCodeSlots;
  uint64_t* oempty = ofull + kOpSlots;
  uint64_t* sfull = oempty + kOpSlots;
  uint64_t* sempty = sfull + kScaleSlots;
  uint64_t* dfull = sempty + kScaleSlots;
  uint64_t* dempty = dfull + 2;
  uint64_t* xready = dempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(xready + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = (int)(((int64_t)N * blockIdx.x) / geo.nblk);
  const int rows = (int)(((int64_t)N * (blockIdx.x + 1)) / geo.nblk) - r0;  // <= R <= 128
  const int nst = K / kStageCodes;
  const int nwin = (ngroups + kWinGroups - 1) / kWinGroups;

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) {
    for (int s = 0; s < geo.ncs; ++s) {
      mbar_init(&cfull[s], 1);
      mbar_init(&cempty[s], kDecWarps);
    }
    for (int s = 0; s < kOpSlots; ++s) {
      mbar_init(&ofull[s], kDecWarps);
      mbar_init(&oempty[s], 1);
    }
    for (int s = 0; s < kScaleSlots; ++s) {
      mbar_init(&sfull[s], 1);
      mbar_init(&sempty[s], 4);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&dfull[s], 1);
      mbar_init(&dempty[s], 4);
    }
    mbar_init(xready, 1);
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(tmem_slot)), "r"(kTmemCols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool failed = false;

  if (warp == kProdWarp) {
    // ------------------------------------------------------------ producer --
    if (elect_one_sync()) {
      prefetch_tmap(&tmW);
      prefetch_tmap(&tmS);
      prefetch_tmap(&tmB);
      const uint32_t ctx = (uint32_t)geo.R * 128u, stx = (uint32_t)geo.R * 64u;
      int cs = 0, cround = 0;
      for (int i = 0; i < nst; ++i) {
        if (i == 4) mbar_wait(xready, 0, err, failed);  // x's loads would otherwise queue behind the stream
        if (i % kSpw == 0) {                             // the window's scales and biases
          const int wi = i / kSpw, ss = wi % kScaleSlots;
          if (wi >= kScaleSlots) mbar_wait(&sempty[ss], ((wi / kScaleSlots) - 1) & 1, err, failed);
          mbar_arrive_expect_tx(&sfull[ss], stx);
          uint8_t* sd = smem + offS + ss * kScaleSlot;
          tma_load_2d(sd, &tmS, &sfull[ss], wi * kWinGroups, r0);
          tma_load_2d(sd + kRows * 32, &tmB, &sfull[ss], wi * kWinGroups, r0);
        }
        if (cround > 0) mbar_wait(&cempty[cs], (cround - 1) & 1, err, failed);
        mbar_arrive_expect_tx(&cfull[cs], ctx);
        tma_load_2d(smem + cs * geo.cslot, &tmW, &cfull[cs], i * 128, r0);
        if (++cs == geo.ncs) { cs = 0; ++cround; }
      }
      // no copy may still be writing shared memory when the CTA exits
      for (int i = max(0, nst - geo.ncs); i < nst; ++i)
        mbar_wait(&cfull[i % geo.ncs], (i / geo.ncs) & 1, err, failed);
      for (int wi = max(0, nwin - kScaleSlots); wi < nwin; ++wi)
        mbar_wait(&sfull[wi % kScaleSlots], (wi / kScaleSlots) & 1, err, failed);
    }
  } else if (warp < kDecWarps) {
    // ------------------------------------------------------- decode warps --
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // x -> f16 pieces in the A operand's k order (e0, e4, e1/16, e5/16, e2, e6,
    // e3/16, e7/16), one power-of-two pre-scale per scale group; group sums
    const int t = threadIdx.x;  // 0 .. 511
    for (int pc = t; pc < K / 8; pc += kDecWarps * 32) {  // the range test is uniform within each group's lanes
      const uint4 xv = __ldg(reinterpret_cast<const uint4*>(x) + pc);
      uint32_t mb = max_mag8(xv);
#pragma unroll
      for (int o = 1; o < kLpg; o <<= 1) mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, o));
      int sigma = 0;
      if (mb != 0) {
        const int E = (int)(mb >> 7);
        const int e = (E == 0) ? (-133 + (31 - __clz((int)(mb & 0x7Fu)))) : (E - 127);
        sigma = min(14 - e, 127);
      }
      const float xs = exp2i_f32(sigma);
      const uint32_t v[4] = {xv.x, xv.y, xv.z, xv.w};
      float f[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        f[2 * j] = bf16_lo(v[j]) * xs;
        f[2 * j + 1] = bf16_hi(v[j]) * xs;
      }
      const uint4 o = make_uint4(f16x2_bits(f[0], f[4]), f16x2_bits(f[1] * 0.0625f, f[5] * 0.0625f),
                                 f16x2_bits(f[2], f[6]), f16x2_bits(f[3] * 0.0625f, f[7] * 0.0625f));
      reinterpret_cast<uint4*>(x16)[pc] = o;
      const __half2* hp = reinterpret_cast<const __half2*>(&o);
      float s1 = 0.f, s2 = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 hf = __half22float2(hp[j]);
        s1 += hf.x + hf.y;
        s2 += (hf.x + hf.y) * ((j & 1) ? 16.0f : 1.0f);
      }
#pragma unroll
      for (int o2 = 1; o2 < kLpg; o2 <<= 1) {
        s1 += __shfl_xor_sync(0xffffffffu, s1, o2);
        s2 += __shfl_xor_sync(0xffffffffu, s2, o2);
      }
      if ((pc & (kLpg - 1)) == 0) {
        const int g = pc / kLpg;
        ginv[g] = exp2i_f32(-sigma);
        gx1[g] = s1;
        gx2[g] = s2;
      }
    }
    asm volatile("bar.sync 1, %0;" :: "n"(kDecWarps * 32) : "memory");
    if (t == 0) mbar_arrive(xready);

    const int q = warp & 3, c = warp >> 2;       // lane quadrant; quarter of the stage's 128-byte row
    const int r = 4 * lane + q;                  // this thread's row (tensor-memory lane 32 q + lane)
    const bool valid = r < rows;
    const uint32_t t_lane = (uint32_t)(32 * q) << 16;
    int cs = 0, cround = 0;
    for (int i = 0; i < nst; ++i) {
      const int os = i % kOpSlots;
      if (i >= kOpSlots) {
        mbar_wait(&oempty[os], ((i / kOpSlots) - 1) & 1, err, failed);  // stage i - 2's MMAs are done
        tc_fence_after();
      }
      // B operand of stage i: 4 blocks (4 k-steps of 16 each) of 16 rows x 128 bytes,
      // 128-byte swizzled; row j of k-step kk holds x iff j is kk's group in the window
      {
        const int u = t;                          // 16-byte piece u of the 8 KB stage
        const int blk = u >> 7, n = (u >> 3) & 15, ch = u & 7;
        const int kk = blk * 4 + (ch >> 1);       // k-step of this piece (16 k per step, 8 per piece)
        const int kglob = i * kStageCodes + kk * 16 + (ch & 1) * 8;
        const int gwin = (kglob / GROUP) % kWinGroups;
        const uint4 val = (n == gwin) ? reinterpret_cast<const uint4*>(x16)[kglob >> 3] : make_uint4(0, 0, 0, 0);
        const uint32_t off = (uint32_t)(blk * 2048 + (n >> 3) * 1024 + (n & 7) * 128 + ((ch ^ (n & 7)) << 4));
        *reinterpret_cast<uint4*>(smem + offB + os * kBStage + off) = val;
      }
      mbar_wait(&cfull[cs], cround & 1, err, failed);
      uint4 p0 = make_uint4(0, 0, 0, 0), p1 = make_uint4(0, 0, 0, 0);
      if (valid) {
        const uint32_t rowa = base + cs * geo.cslot + (uint32_t)r * 128u;
        p0 = lds128(rowa + (uint32_t)(((2 * c) ^ (r & 7)) << 4));
        p1 = lds128(rowa + (uint32_t)(((2 * c + 1) ^ (r & 7)) << 4));
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&cempty[cs]);
      const uint32_t wv[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
      uint32_t a[32];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t w8 = wv[j] >> 8;
        a[4 * j] = (wv[j] & 0x000F000Fu) | 0x64006400u;
        a[4 * j + 1] = (wv[j] & 0x00F000F0u) | 0x64006400u;
        a[4 * j + 2] = (w8 & 0x000F000Fu) | 0x64006400u;
        a[4 * j + 3] = (w8 & 0x00F000F0u) | 0x64006400u;
      }
      asm volatile(
          "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
          "%13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
          :: "r"(tmem + t_lane + kAcol + 128u * os + 32u * c), "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]),
             "r"(a[4]), "r"(a[5]), "r"(a[6]), "r"(a[7]), "r"(a[8]), "r"(a[9]), "r"(a[10]), "r"(a[11]), "r"(a[12]),
             "r"(a[13]), "r"(a[14]), "r"(a[15]), "r"(a[16]), "r"(a[17]), "r"(a[18]), "r"(a[19]), "r"(a[20]),
             "r"(a[21]), "r"(a[22]), "r"(a[23]), "r"(a[24]), "r"(a[25]), "r"(a[26]), "r"(a[27]), "r"(a[28]),
             "r"(a[29]), "r"(a[30]), "r"(a[31])
          : "memory");
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      tc_fence_before();
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the B bytes, for the MMA
      __syncwarp();
      if (lane == 0) mbar_arrive(&ofull[os]);
      if (++cs == geo.ncs) { cs = 0; ++cround; }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer --
    if (elect_one_sync()) {
      for (int i = 0; i < nst; ++i) {
        const int os = i % kOpSlots;
        const int wi = i / kSpw, p = i % kSpw, db = wi & 1;
        if (p == 0 && wi >= 2) mbar_wait(&dempty[db], ((wi >> 1) - 1) & 1, err, failed);
        mbar_wait(&ofull[os], (i / kOpSlots) & 1, err, failed);
        tc_fence_after();
        const uint32_t bbase = base + offB + os * kBStage;
#pragma unroll
        for (int kk = 0; kk < kStageCodes / 16; ++kk) {
          const uint64_t bdesc = desc_sw128(bbase + (kk >> 2) * 2048) + (uint64_t)(2 * (kk & 3));
          const uint32_t acc = (p > 0 || kk > 0) ? 1u : 0u;
          asm volatile(
              "{\n\t.reg .pred pp;\n\tsetp.ne.u32 pp, %4, 0;\n\t"
              "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, pp;\n\t}"
              :: "r"(tmem + kDcol + 32u * db), "r"(tmem + kAcol + 128u * os + 8u * kk), "l"(bdesc), "r"(kIdesc),
                 "r"(acc)
              : "memory");
        }
        tc_commit(&oempty[os]);
        if (p == kSpw - 1 || i == nst - 1) tc_commit(&dfull[db]);
      }
    }
  } else {
    // -------------------------------------------------------------- epilogue --
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int q = warp & 3;
    const int r = 4 * lane + q;
    const bool valid = r < rows;
    float yacc = 0.f;
    for (int wi = 0; wi < nwin; ++wi) {
      const int db = wi & 1, ss = wi % kScaleSlots;
      mbar_wait(&dfull[db], (wi >> 1) & 1, err, failed);
      mbar_wait(&sfull[ss], (wi / kScaleSlots) & 1, err, failed);
      tc_fence_after();
      uint32_t d[16];
      asm volatile(
          "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
          : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3]), "=r"(d[4]), "=r"(d[5]), "=r"(d[6]), "=r"(d[7]),
            "=r"(d[8]), "=r"(d[9]), "=r"(d[10]), "=r"(d[11]), "=r"(d[12]), "=r"(d[13]), "=r"(d[14]), "=r"(d[15])
          : "r"(tmem + ((uint32_t)(32 * q) << 16) + kDcol + 32u * db));
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&dempty[db]);
      if (valid) {
        const uint32_t sa = base + offS + ss * kScaleSlot + (uint32_t)r * 32u;
        const uint4 s0 = lds128(sa), s1 = lds128(sa + 16), b0 = lds128(sa + kRows * 32), b1 = lds128(sa + kRows * 32 + 16);
        const uint32_t sw[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
        const uint32_t bw[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
        const int gn = min(kWinGroups, ngroups - wi * kWinGroups);
#pragma unroll
        for (int j = 0; j < kWinGroups; ++j) {
          if (j < gn) {
            const int g = wi * kWinGroups + j;
            const float sj = (j & 1) ? bf16_hi(sw[j >> 1]) : bf16_lo(sw[j >> 1]);
            const float bj = (j & 1) ? bf16_hi(bw[j >> 1]) : bf16_lo(bw[j >> 1]);
            yacc = fmaf(fmaf(sj, __uint_as_float(d[j]) - 1024.f * gx1[g], bj * gx2[g]), ginv[g], yacc);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sempty[ss]);
    }
    if (valid) y[r0 + r] = (uint16_t)f32_to_bf16_rn(yacc);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(kTmemCols) : "memory");
  }
}

// The plan: one CTA per SM (R = ceil(N / SMs) <= 128 rows), K a multiple of the
// 256-code stage, as many code slots as fit.
bool plan_affine(const DevInfo& d, int64_t N, int64_t K, int group, AffGeo* g) {
  if (K > kMaxK || K % kStageCodes != 0 || K % group != 0 || d.sm_count < 1) return false;
  if (group != 32 && group != 64 && group != 128) return false;
  if ((K / group) % 8 != 0) return false;  // 16-byte scale rows for the TMA boxes
  const int64_t nblk = std::min<int64_t>(d.sm_count, N);
  const int64_t R = (N + nblk - 1) / nblk;
  if (R < 1 || R > kRows) return false;
  g->nblk = (int)nblk;
  g->R = (int)R;
  g->cslot = (uint32_t)((R + 7) / 8) * 1024u;
  const uint32_t fixed = 1024u + fixed_bytes((int)K, group);
  if (fixed >= kSmemBytes) return false;
  const uint32_t ncs = std::min<uint32_t>(kMaxCodeSlots, (kSmemBytes - fixed) / g->cslot);
  if (ncs < 3) return false;
  g->ncs = (int)ncs;
  return true;
}

bool make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* p, uint64_t inner, uint64_t rows,
              uint64_t pitch, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle sw) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {pitch};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(p), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int GROUP>
cudaError_t launch_group(const DevInfo& d, const AffGeo& geo, const uint16_t* x, const uint32_t* w,
                         const uint16_t* scales, const uint16_t* biases, int64_t N, int64_t K, uint16_t* y,
                         cudaStream_t s) {
  CUtensorMap tw, ts, tb;
  const uint64_t groups = (uint64_t)(K / GROUP);
  if (!make_map(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, (uint64_t)K / 2, (uint64_t)N, (uint64_t)K / 2, 128,
                (uint32_t)geo.R, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&ts, CU_TENSOR_MAP_DATA_TYPE_UINT16, scales, groups, (uint64_t)N, groups * 2, kWinGroups,
                (uint32_t)geo.R, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !make_map(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT16, biases, groups, (uint64_t)N, groups * 2, kWinGroups,
                (uint32_t)geo.R, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  cudaError_t e =
      cudaFuncSetAttribute(qmv_affine_kernel<GROUP>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)geo.nblk);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, qmv_affine_kernel<GROUP>, tw, ts, tb, x, (int)N, (int)K, geo, y, d.err);
}

}  // namespace

bool qmv_affine_supported(const DevInfo& d, int64_t N, int64_t K, int group) {
  AffGeo g;
  return plan_affine(d, N, K, group, &g);
}

cudaError_t launch_qmv_affine(const DevInfo& d, const uint16_t* x, const uint32_t* w, const uint16_t* scales,
                              const uint16_t* biases, int64_t N, int64_t K, int group, uint16_t* y,
                              cudaStream_t s) {
  AffGeo g;
  if (!plan_affine(d, N, K, group, &g)) return cudaErrorInvalidValue;
  if (group == 32) return launch_group<32>(d, g, x, w, scales, biases, N, K, y, s);
  if (group == 64) return launch_group<64>(d, g, x, w, scales, biases, N, K, y, s);
  if (group == 128) return launch_group<128>(d, g, x, w, scales, biases, N, K, y, s);
  return cudaErrorInvalidValue;
}

}  // namespace fp4
