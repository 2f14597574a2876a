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
// written as kTerms NVFP4 terms in radix 4, block by block (16 elements):
//     x = 2^e0 * S_b * (sum_t d_t 4^-t + r),   d_t in {-2, ..., 2},
// with 2^e0 a per-vector power of two (max|x| / 2^e0 in [256, 512)) and S_b a
// power of two per block chosen so |x| / (2^e0 S_b) <= 2: then
// d_0 = rint(v), v <- 4 (v - d_0), ... keeps every digit in [-2, 2] (exact
// e2m1 codes) and each term's block scale S_b 4^-t is an exact E4M3 value.
// Eight terms carry 16 bits per block -- |r| <= 2^-15 of the block scale,
// about 2^-13 of a typical element -- and become rows 0..7 of the B operand.  The MMA
// yields D[row, t] = sum_k W[row, k] (d_t S_b 4^-t)[k] in fp32 tensor memory;
// the epilogue forms y = gs_w 2^e0 sum_t D[row, t].
//
// One CTA per SM owns <= 128 consecutive rows (row ranges balanced to +-1).
//   warp 0: TMA producer -- 8-row atoms of W (128-byte swizzle) per K = 256
//           stage, into a 6-stage ring, issued before griddepcontrol.wait
//           (programmatic dependent launch: no earlier kernel writes W);
//   warp 1: tensor memory allocation; one thread copies each stage's scale
//           tiles to tensor memory (tcgen05.cp) and issues 4 MMAs (M 128,
//           N 16, K 64) into four independent accumulators;
//   warps 2-17: four groups of four warps; group g prepares stages
//           kb % 4 == g -- permute the weights' linear E4M3 scales into the
//           128x4 tile order tcgen05.cp reads, copy the < 8 rows that do not
//           fill a TMA atom, and build the x terms (codes + scales); after the
//           last stage group 0 reads D and writes y.
// The B operand's rows 8-15 are the next stage's term atom (128-byte-swizzle
// stride 1024); their block scales are zero, so they add nothing.
#include <algorithm>
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "launch.h"

namespace fp4 {

namespace {

constexpr int kTerms = 8;           // x expansion terms (B rows 0..7, one 1 KB atom)
constexpr int kStages = 6;          // W / scale-tile / term ring
constexpr int kRawDepth = 12;       // ring of the prep warps' own copies (scales, partial-atom rows)
constexpr int kAhead = 8;           // their lookahead (a multiple of kGroups), independent of MMA progress
constexpr uint32_t kRawBytes = 128 * 16 + 8 * 128;  // 128 rows x 16 scale bytes + up to 8 rows x 128 B
constexpr int kBK = 256;            // codes per stage (128 bytes per row)
constexpr int kRows = 128;          // rows per CTA at most (one M = 128 tile)
constexpr int kGroups = 4;          // prep groups; group g prepares stages kb % kGroups == g
constexpr int kGroupThreads = 128;  // one group = 4 warps, two elements per thread per stage
constexpr int kPrep = kGroups * kGroupThreads;
constexpr int kThreads = 64 + kPrep;  // TMA warp, MMA warp, prep warps (group 0 also runs the epilogue)
constexpr uint32_t kWBytes = kRows * 128;  // 16 KB
constexpr uint32_t kSFBytes = 4 * 512;     // four 128x4 scale tiles (one per MMA k-step)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfCol = 64;            // D: four accumulators of 16 columns, [0, 64)
// kind::mxf4nvf4 descriptor: E2M1 A/B, K-major, N = 16, E4M3 scales, M = 128
constexpr uint32_t kIdesc = (1u << 7) | (1u << 10) | ((16u >> 3) << 17) | ((128u >> 4) << 24);

// shared memory offsets (from a 1024-aligned base)
constexpr uint32_t kOffW = 0;
constexpr uint32_t kOffB = kOffW + kStages * kWBytes;            // (kStages + 1) term atoms of 1 KB
constexpr uint32_t kOffSFA = kOffB + (kStages + 1) * 1024;
constexpr uint32_t kOffSFB = kOffSFA + kStages * kSFBytes;
constexpr uint32_t kOffRaw = kOffSFB + kStages * kSFBytes;       // kRawDepth x kRawBytes
constexpr uint32_t kOffX = kOffRaw + kRawDepth * kRawBytes;        // x (bf16), K <= kMaxK
constexpr int kMaxK = 16384 + 1024;                               // 17408
constexpr uint32_t kOffBar = kOffX + kMaxK * 2;
constexpr uint32_t kSmemBytes = kOffBar + 256 + 1024;

__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(sbo >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
__device__ __forceinline__ uint64_t desc_sf(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(128 >> 4) << 32) | ((uint64_t)1 << 46);
}
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

__global__ void __launch_bounds__(kThreads, 1) qmv_tc_kernel(const __grid_constant__ CUtensorMap tmW,
                                                              const uint16_t* __restrict__ x,
                                                              const uint32_t* __restrict__ w,
                                                              const uint8_t* __restrict__ scales,
                                                              const float* __restrict__ gs_w, int N, int K,
                                                              uint16_t* __restrict__ y, unsigned* __restrict__ err) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* empty = full + kStages;
  uint64_t* done = empty + kStages;
  uint64_t* xbar = done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(xbar + 1);
  float* red = reinterpret_cast<float*>(tmem_slot + 4);  // kPrep / 32 floats
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem + kOffX);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = (int)(((int64_t)N * blockIdx.x) / gridDim.x);
  const int r1 = (int)(((int64_t)N * (blockIdx.x + 1)) / gridDim.x);
  const int rows = r1 - r0;                  // <= 128
  const int atoms = rows >> 3, rem = rows & 7;
  const int nkb = K / kBK;
  const int words = K >> 3;

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1 + kGroupThreads);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    mbar_init(xbar, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(tmem_slot)), "r"(kTmemCols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // rows 8..15 of every stage's term scale tiles stay zero (those B rows add nothing)
  for (uint32_t i = threadIdx.x; i < kStages * kSFBytes / 4; i += kThreads)
    reinterpret_cast<uint32_t*>(smem + kOffSFB)[i] = 0u;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool failed = false;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer (weights)
    if (elect_one_sync()) {
      prefetch_tmap(&tmW);
      for (int kb = 0; kb < nkb; ++kb) {
        const int s = kb % kStages, round = kb / kStages;
        if (round > 0) mbar_wait(&empty[s], (round - 1) & 1, err, failed);
        mbar_arrive_expect_tx(&full[s], (uint32_t)atoms * 1024u);
        uint8_t* st = smem + kOffW + s * kWBytes;
        for (int a = 0; a < atoms; ++a) tma_load_2d(st + a * 1024, &tmW, &full[s], kb * 128, r0 + 8 * a);
      }
      for (int k = std::max(0, nkb - kStages); k < nkb; ++k)
        mbar_wait(&full[k % kStages], (k / kStages) & 1, err, failed);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    if (elect_one_sync()) {
      for (int kb = 0; kb < nkb; ++kb) {
        const int s = kb % kStages;
        mbar_wait(&full[s], (kb / kStages) & 1, err, failed);
        tc_fence_after();
        const uint32_t sfa_t = tmem + kSfCol + s * 32, sfb_t = sfa_t + 16;
        const uint32_t sfa_s = base + kOffSFA + s * kSFBytes, sfb_s = base + kOffSFB + s * kSFBytes;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" :: "r"(sfa_t + 4 * j), "l"(desc_sf(sfa_s + 512 * j)) : "memory");
          asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" :: "r"(sfb_t + 4 * j), "l"(desc_sf(sfb_s + 512 * j)) : "memory");
        }
        const uint64_t adesc = desc_sw128(base + kOffW + s * kWBytes, 1024);
        const uint64_t bdesc = desc_sw128(base + kOffB + s * 1024, 1024);  // rows 8-15: next term atom
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          // k-step j accumulates into its own 16-column tile, so the four MMAs of a
          // stage do not wait on each other; the epilogue adds the four tiles
          const uint32_t acc = (kb > 0) ? 1u : 0u;
          asm volatile(
              "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %6, 0;\n\t"
              "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
              :: "r"(tmem + 16 * j), "l"(adesc + (uint64_t)(2 * j)), "l"(bdesc + (uint64_t)(2 * j)), "r"(kIdesc),
                 "r"(sfa_t + 4 * j), "r"(sfb_t + 4 * j), "r"(acc) : "memory");
        }
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                     :: "r"(smem_u32(&empty[s])) : "memory");
      }
      asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                   :: "r"(smem_u32(done)) : "memory");
    }
  } else {
    // ------------------------------------------- prep warps (2..17), then epilogue
    const int pa = threadIdx.x - 64;           // 0..kPrep-1
    const int grp = pa / kGroupThreads;        // prep group
    const int pt = pa % kGroupThreads;         // thread within the group
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // x (bf16, K*2 bytes) -> shared memory in one bulk copy, then max|x| from shared memory
    if (pa == 0) {
      mbar_arrive_expect_tx(xbar, (uint32_t)K * 2u);
      bulk_load(xs, x, (uint32_t)K * 2u, xbar);
    }
    mbar_wait(xbar, 0, err, failed);
    uint32_t m2 = 0;
    for (int v = pa; v < words; v += kPrep) {
      const uint4 q = reinterpret_cast<const uint4*>(xs)[v];
      m2 = __vmaxu2(m2, q.x & 0x7FFF7FFFu);
      m2 = __vmaxu2(m2, q.y & 0x7FFF7FFFu);
      m2 = __vmaxu2(m2, q.z & 0x7FFF7FFFu);
      m2 = __vmaxu2(m2, q.w & 0x7FFF7FFFu);
    }
    uint32_t mb = max(m2 & 0xFFFFu, m2 >> 16);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, o));
    if (lane == 0) red[pa >> 5] = __uint_as_float(mb << 16);
    asm volatile("bar.sync 1, %0;" :: "n"(kPrep) : "memory");  // prep warps only
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < kPrep / 32; ++i) amax = fmaxf(amax, red[i]);
    // e0: max|x| / 2^e0 in [256, 512), so every block scale S_b = 2^k fits k <= 8
    int e0 = 0;
    if (amax > 0.f) {
      int ex;
      frexpf(amax, &ex);  // amax = m * 2^ex, 0.5 <= m < 1
      e0 = max(ex - 9, -126);
    }
    const float pre = ldexpf(1.0f, -e0);

    const int b16 = pt >> 3;  // this thread's 16-element block within the stage (0..15)
    // The prep warps' global traffic -- row pt's 16 linear scale bytes and, for
    // threads < 8*rem, one 16-byte piece of the rows that do not fill a TMA atom --
    // runs kAhead stages ahead through a private cp.async ring.  Every thread later
    // reads back only what it copied itself, so the ring needs no barrier and never
    // waits for the MMA.
    auto issue = [&](int kb) {
      const uint32_t slot = base + kOffRaw + (kb % kRawDepth) * kRawBytes;
      if (pt < rows) {
        const uint8_t* src = scales + (int64_t)(r0 + pt) * (K >> 4) + kb * 16;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(slot + pt * 16), "l"(src) : "memory");
      }
      if (pt < rem * 8) {
        const uint8_t* src = reinterpret_cast<const uint8_t*>(w) + (int64_t)(r0 + 8 * atoms + (pt >> 3)) * (K >> 1) +
                             kb * 128 + (pt & 7) * 16;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(slot + 2048 + pt * 16), "l"(src) : "memory");
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
    };
    // this group's stages are grp, grp + kGroups, ...; its copies run kAhead/kGroups of them ahead
    constexpr int kAheadG = kAhead / kGroups;
    int issued = grp;
    for (int p = 0; p < kAheadG; ++p) {
      if (issued < nkb) issue(issued);
      else asm volatile("cp.async.commit_group;" ::: "memory");
      issued += kGroups;
    }
    for (int kb = grp; kb < nkb; kb += kGroups) {
      const int s = kb % kStages, round = kb / kStages;
      if (issued < nkb) issue(issued);
      else asm volatile("cp.async.commit_group;" ::: "memory");  // keep the group count uniform
      issued += kGroups;
      asm volatile("cp.async.wait_group %0;" :: "n"(kAheadG) : "memory");  // this thread's copies for kb
      const uint8_t* rawp = smem + kOffRaw + (kb % kRawDepth) * kRawBytes;
      if (round > 0) mbar_wait(&empty[s], (round - 1) & 1, err, failed);  // stage slot s is free
      // (a) weight scales of row pt: 16 E4M3 bytes -> word j of tile j, 16B-row (pt%32), slot pt/32
      uint8_t* sfa = smem + kOffSFA + s * kSFBytes;
      uint4 sv = make_uint4(0, 0, 0, 0);
      if (pt < rows) sv = *reinterpret_cast<const uint4*>(rawp + pt * 16);
      const uint32_t so = (uint32_t)((pt & 31) * 16 + (pt >> 5) * 4);
      *reinterpret_cast<uint32_t*>(sfa + 0 * 512 + so) = sv.x;
      *reinterpret_cast<uint32_t*>(sfa + 1 * 512 + so) = sv.y;
      *reinterpret_cast<uint32_t*>(sfa + 2 * 512 + so) = sv.z;
      *reinterpret_cast<uint32_t*>(sfa + 3 * 512 + so) = sv.w;
      // (a') the partial atom's piece this thread copied, into the swizzled W tile
      if (pt < rem * 8) {
        const int rr = pt >> 3, c = pt & 7;
        *reinterpret_cast<uint4*>(smem + kOffW + s * kWBytes + atoms * 1024 + rr * 128 + ((c ^ rr) << 4)) =
            *reinterpret_cast<const uint4*>(rawp + 2048 + pt * 16);
      }
      // (b) x terms for elements 2pt, 2pt+1 of this stage (radix-4 digits, see the header)
      const uint32_t xv = *reinterpret_cast<const uint32_t*>(xs + kb * kBK + 2 * pt);
      const float R0 = bf16_lo(xv) * pre, R1 = bf16_hi(xv) * pre;
      float mb = fmaxf(fabsf(R0), fabsf(R1));
      mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
      mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
      mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 4));
      // S_b = 2^kexp with mb < 2^(kexp+1), 5 <= kexp <= 8: the floor keeps the last
      // term's scale 2^(kexp-14) >= 2^-9, the smallest E4M3 value; a block that small
      // (< 1/8 of max|x|) then carries a few bits less of its own, which is below
      // 2^-18 of max|x|
      int kexp = 5;
      if (mb > 0.f) {
        int ex;
        frexpf(mb, &ex);  // mb < 2^ex
        kexp = min(max(ex - 1, 5), 8);
      }
      const float invS = ldexpf(1.0f, -kexp);
      float v0 = R0 * invS, v1 = R1 * invS;
      uint8_t* batom = smem + kOffB + s * 1024;
      uint8_t* sfb = smem + kOffSFB + s * kSFBytes;
#pragma unroll
      for (int t = 0; t < kTerms; ++t) {
        // round to the nearest integer (ties to even): |v| <= 2, so adding 1.5 * 2^23 leaves
        // exactly the rounded value's bits in the low mantissa; subtracting it back is exact
        const float d0 = __fsub_rn(__fadd_rn(v0, 12582912.0f), 12582912.0f);
        const float d1 = __fsub_rn(__fadd_rn(v1, 12582912.0f), 12582912.0f);
        const uint32_t code = e2m1x2_rn(d0, d1);  // exact: digits in [-2, 2]
        v0 = (v0 - d0) * 4.0f;
        v1 = (v1 - d1) * 4.0f;
        // byte pt of term row t, 128-byte swizzle within the 1 KB atom
        batom[t * 128 + ((((pt >> 4) ^ t) & 7) << 4) + (pt & 15)] = (uint8_t)code;
        if ((pt & 7) == 0) {
          const int e = kexp - 2 * t;  // term scale 2^e, -9 <= e <= 8, as an E4M3 byte
          const uint32_t sb = (e >= -6) ? (uint32_t)((e + 7) << 3) : (1u << (e + 9));
          sfb[(b16 >> 2) * 512 + t * 16 + (b16 & 3)] = (uint8_t)sb;
        }
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive(&full[s]);
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    // ---- epilogue (group 0, warps 2..5 = lane quadrants 2, 3, 0, 1): y = gs_w 2^e0 sum_t D[row, t]
    if (grp == 0) {
    mbar_wait(done, 0, err, failed);
    tc_fence_after();
    const int q = warp & 3;
    float dsum[kTerms];
#pragma unroll
    for (int t = 0; t < kTerms; ++t) dsum[t] = 0.f;
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      uint32_t d[16];
      asm volatile(
          "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
          : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3]), "=r"(d[4]), "=r"(d[5]), "=r"(d[6]), "=r"(d[7]),
            "=r"(d[8]), "=r"(d[9]), "=r"(d[10]), "=r"(d[11]), "=r"(d[12]), "=r"(d[13]), "=r"(d[14]), "=r"(d[15])
          : "r"(tmem + ((uint32_t)(32 * q) << 16) + 16 * a));
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
      for (int t = 0; t < kTerms; ++t) dsum[t] += __uint_as_float(d[t]);
    }
    const int row = 32 * q + lane;
    if (row < rows) {
      float acc = 0.f;
#pragma unroll
      for (int t = kTerms - 1; t >= 0; --t) acc += dsum[t];
      const float g = gs_w ? __ldg(gs_w) : 1.0f;
      y[r0 + row] = (uint16_t)f32_to_bf16_rn(ldexpf(acc, e0) * g);
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

}  // namespace

// Whether the tensor-core GEMV handles this NVFP4 problem (else the mma.sync kernel does).
bool qmv_tc_supported(const DevInfo& d, int64_t N, int64_t K) {
  return K % kBK == 0 && K <= kMaxK && N >= 1 && (N + kRows - 1) / kRows <= d.sm_count &&
         kSmemBytes <= d.smem_optin;
}

cudaError_t launch_qmv_tc(const DevInfo& d, const uint16_t* x, const uint32_t* w, const uint8_t* scales,
                          const float* gs_w, int64_t N, int64_t K, uint16_t* y, cudaStream_t s) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorInvalidValue;
  CUtensorMap tm;
  cuuint64_t dims[2] = {(cuuint64_t)(K / 2), (cuuint64_t)N};
  cuuint64_t strides[1] = {(cuuint64_t)(K / 2)};
  cuuint32_t box[2] = {128, 8};
  cuuint32_t estr[2] = {1, 1};
  if (fn(&tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint32_t*>(w), dims, strides, box, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(qmv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  const int64_t grid = std::min<int64_t>(N, std::max<int64_t>(d.sm_count, (N + kRows - 1) / kRows));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, qmv_tc_kernel, tm, x, w, scales, gs_w, (int)N, (int)K, y, d.err);
}

}  // namespace fp4
