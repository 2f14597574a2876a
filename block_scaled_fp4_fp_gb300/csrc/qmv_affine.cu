// qmv_affine.cu -- affine 4-bit decode GEMV (group 32 / 64 / 128, bf16 scale
// and bias) fed by a TMA shared-memory ring, multiplied with mma.sync.
//
// Pages: "epic: NVIDIA Volta (sm_70) inference acceleration program #1536"
// (Baseline: the decode step streams affine 4-bit group-64 weights at 7.7 % of
// the V100's bandwidth, ALU-bound; Diagnosis 3: the accumulator type -- fp32
// here), "mlx 0.30.7.3 -> 0.30.7.6" quantized.cpp (affine w = q * scale + bias).
//
// y[n] = sum_g s[n,g] (sum_{k in g} q[n,k] x[k]) + b[n,g] X_g.  The weight
// stream is the cost; the kernel is built so the consumers keep up with it:
//   * warp 16 (one thread) streams W by TMA: per stage of KS = 128 IPS codes
//     (IPS = 4, 8 or 16 item columns, the widest whose ring still holds three
//     slots) KS / 256 boxes of R rows x 128 bytes (128-byte swizzle) plus one box
//     of R rows of scales and one of biases, into a ring of slots.  The first kXPre stages go out before the
//     previous kernel has finished (programmatic dependent launch: no kernel of
//     this library writes weights and releases its dependents early); later ones
//     wait until x has been staged, whose loads would otherwise queue behind them;
//   * warps 0-15 decode and multiply with mma.sync m16n8k16 (f16 inputs, fp32
//     accumulation), W as the A operand: lane (g, t) = (lane / 4, lane % 4)
//     holds chunk t (32 codes) of rows g and g + 8 of a 16-row group, so one MMA
//     covers 16 rows x 16 codes.  A code pair becomes an f16 pair with one LOP3:
//     (w & 0x000F000F) | 0x64006400 = f16(1024 + q) for nibbles 0 and 4,
//     (w & 0x00F000F0) | 0x64006400 = f16(1024 + 16 q) for nibbles 1 and 5, the
//     same on w >> 8 for nibbles 2, 6 and 3, 7 (five instructions per eight
//     codes).  B is x: column i holds chunk i's x at lane t = i's k positions
//     (zeros elsewhere), staged as f16 in the decode's pair order with the
//     nibble-1/3 elements divided by 16, so column i of D is chunk i's
//     1024 X'_i + sum q x for each row -- every D element inside one scale group;
//   * x carries one power-of-two pre-scale per scale group (max|x| 2^sigma in
//     [2^14, 2^15): every bf16 value is exact in f16 down to 2^-24 of the group's
//     max); per chunk (groups of 32) or chunk pair (64, 128) the kernel keeps
//     P = 2^-sigma, Q = 1024 P X' and Z = P X, so a row's pair adds
//     s (P (D0 + D1) - Q) + b Z;
//   * warp w takes item column jj = w % IPS (128 codes) of every stage for the
//     row groups w / IPS, w / IPS + 16 / IPS, ..., so its x fragments load once
//     per stage, its items are independent (instruction-level parallelism) and
//     its accumulators stay in registers; the partial row sums meet
//     in shared memory and are added in item-column order (deterministic).
// Every mbarrier wait is bounded (an expired wait records FP4_ERR_TIMEOUT).
#include <algorithm>
#include <cstring>
#include <mutex>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "launch.h"

namespace fp4 {

namespace {

constexpr int kCWarps = 16;                   // consumer warps
constexpr int kThreads = (kCWarps + 1) * 32;  // + the TMA producer warp
constexpr int kMaxK = 32768;                  // a CTA stages its whole x slice in shared memory
constexpr int kMaxRows = 256;                 // rows per CTA (TMA box height)
constexpr int kMaxSlots = 24;
constexpr int kXPre = 4;                      // stages issued before x has been staged
constexpr uint32_t kSmemBytes = 227u * 1024u;
constexpr uint32_t kBarBytes = 512;
constexpr uint32_t kPartBytes = 16 * kMaxRows * 4;  // [item column][row] partial sums
constexpr int kMaxSplit = 4;                        // CTAs per cluster (K slices) at most
constexpr uint32_t kXPartBytes = kMaxSplit * kMaxRows * 4;  // rank 0: the other ranks' row partials
static_assert(2 * kMaxSlots + 3 <= kBarBytes / 8, "barrier area");

// A stage is IPS item columns of 128 codes (KS = 128 IPS codes per row); IPS is
// chosen per launch (4, 8 or 16: wider stages give each warp several independent
// items when a CTA has few rows) with KS >= 8 GROUP (16-byte scale boxes).
template <int GROUP, int IPS_> struct AffCfg {
  static constexpr int IPS = IPS_;
  static constexpr int KS = 128 * IPS;                          // codes per stage
  static constexpr int WR = kCWarps / IPS;                      // warps per item column
  static constexpr int RGW = 16 / WR;                           // row groups per warp at most
  static constexpr bool kPairs = GROUP >= 64;                   // chunk pairs share a scale group
  static_assert(KS >= 8 * GROUP, "a stage holds at least 8 scale groups");
};

// m16n8k16, W rows g and g + 8 as A, x as B
__device__ __forceinline__ void mma_wa(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                       uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}

__device__ __forceinline__ float4 lds128f(uint32_t a) {
  const uint4 v = lds128(a);
  return make_float4(__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z), __uint_as_float(v.w));
}

// shared::cluster address of a shared-memory location in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t mapa_u32(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

__device__ __forceinline__ float lds_bf16(uint32_t a) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
  return __uint_as_float((uint32_t)v << 16);
}

__device__ __forceinline__ uint32_t f16x2_bits(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// one 32-bit word of eight codes -> the four f16 pairs of the plan above
__device__ __forceinline__ void decode_word(uint32_t w, uint32_t* p) {
  const uint32_t w8 = w >> 8;
  p[0] = (w & 0x000F000Fu) | 0x64006400u;   // 1024 + q0, 1024 + q4
  p[1] = (w & 0x00F000F0u) | 0x64006400u;   // 1024 + 16 q1, 1024 + 16 q5
  p[2] = (w8 & 0x000F000Fu) | 0x64006400u;  // 1024 + q2, 1024 + q6
  p[3] = (w8 & 0x00F000F0u) | 0x64006400u;  // 1024 + 16 q3, 1024 + 16 q7
}

struct AffGeo {
  int nblk = 0;        // CTAs (row blocks)
  int R = 0;           // rows per CTA at most (blocks own R or R - 1)
  int RG = 0;          // 16-row groups per CTA
  int nslots = 0;      // ring slots
  uint32_t cb = 0;     // bytes of one code box region (RG * 16 rows * 128 B)
  uint32_t sbytes = 0; // scale (and bias) bytes per row per stage
  uint32_t slot = 0;   // bytes per slot
};

// Shared memory (from a 1024-aligned base): [ring | x f16 (K) | 64 zero bytes |
// per-chunk or per-pair constants (float4) | partial sums | barriers].
__host__ __device__ inline uint32_t x_region_bytes(int K, int group) {
  const uint32_t nconst = (uint32_t)(group >= 64 ? K / 64 : K / 32);
  return (uint32_t)K * 2u + 64u + nconst * 16u;
}

// The matrices of one launch (as the FP4 GEMV's table): a plain GEMV is a group
// of one; a grouped launch multiplies the same x by up to four matrices of the
// same K and group.  Matrix m owns row blocks blk0[m] .. blk0[m+1]-1, its rows
// dealt out evenly over them.
constexpr int kMaxGroup = 4;
struct AffGroup {
  CUtensorMap tmW[kMaxGroup];  // codes [N_m, K/2] bytes, boxes of R rows x 128 bytes
  CUtensorMap tmS[kMaxGroup];  // bf16 scales [N_m, K/GROUP], boxes of R rows x KS/GROUP
  CUtensorMap tmB[kMaxGroup];  // bf16 biases, the same boxes
  uint16_t* y[kMaxGroup];
  int N[kMaxGroup];
  int blk0[kMaxGroup + 1];
  int count;
};
// The launch that follows on the stream, if the caller names it: once all of a
// CTA's own weights have landed, its producer warms L2 with the first `stages`
// stages the same-numbered CTA of that launch will read (its own maps, stage
// width ks codes).  A hint only: nothing is written.
struct AffNext {
  CUtensorMap tmW[kMaxGroup];
  CUtensorMap tmS[kMaxGroup];
  CUtensorMap tmB[kMaxGroup];
  int N[kMaxGroup];
  int blk0[kMaxGroup + 1];
  int count, ks, nst, split, stages;  // count 0: no prefetch; ks codes per stage, nst stages of K, split ranks
};

template <int GROUP, int IPS_>
__global__ void __launch_bounds__(kThreads, 1) qmv_affine_kernel(
    const __grid_constant__ AffGroup mats, const __grid_constant__ AffNext next, const uint16_t* __restrict__ x,
    int K, int split, AffGeo geo, unsigned* __restrict__ err) {
  using CF = AffCfg<GROUP, IPS_>;
  constexpr int KS = CF::KS, IPS = CF::IPS, WR = CF::WR, RGW = CF::RGW;
  constexpr int kLpg = GROUP / 32;  // 32-code chunks per group
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  // K split: a cluster of `split` CTAs owns a row block; rank q takes stages
  // kb0 .. kb0 + nst - 1 and stages x only over them (kslice codes at most)
  const int rank = (int)(blockIdx.x % (unsigned)split), blk = (int)(blockIdx.x / (unsigned)split);
  const int nst_all = K / KS;
  const int kb0 = (int)(((int64_t)nst_all * rank) / split);
  const int nst = (int)(((int64_t)nst_all * (rank + 1)) / split) - kb0;
  const int kslice = (nst_all + split - 1) / split * KS;
  const int C = (nst * KS) >> 5;  // x chunks of this rank
  const uint32_t ring_bytes = (uint32_t)geo.nslots * geo.slot;
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem + ring_bytes);
  uint4* zero16 = reinterpret_cast<uint4*>(smem + ring_bytes + (uint32_t)kslice * 2u);
  float4* cst = reinterpret_cast<float4*>(smem + ring_bytes + (uint32_t)kslice * 2u + 64u);
  float* part = reinterpret_cast<float*>(smem + ring_bytes + x_region_bytes(kslice, GROUP));
  float* xpart = part + kPartBytes / 4;  // rank 0: [rank][row] partials of the other ranks
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + ring_bytes + x_region_bytes(kslice, GROUP) + kPartBytes +
                                               kXPartBytes);
  uint64_t* empty = full + kMaxSlots;
  uint64_t* xready = empty + kMaxSlots;
  uint64_t* pbar = xready + 1;  // rank 0: the other ranks' partials have landed (byte count)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int mi = 0;  // this CTA's matrix
  while (mi + 1 < mats.count && blk >= mats.blk0[mi + 1]) ++mi;
  const int lb = blk - mats.blk0[mi], nb = mats.blk0[mi + 1] - mats.blk0[mi];
  const int r0 = (int)(((int64_t)mats.N[mi] * lb) / nb);
  const int rows = (int)(((int64_t)mats.N[mi] * (lb + 1)) / nb) - r0;  // <= R
  const CUtensorMap* tmW = &mats.tmW[mi];
  const CUtensorMap* tmS = &mats.tmS[mi];
  const CUtensorMap* tmB = &mats.tmB[mi];
  constexpr int nbox = KS / 256;

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) {
    for (int s = 0; s < geo.nslots; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kCWarps);
    }
    mbar_init(xready, 1);
    mbar_init(pbar, 1);
    fence_barrier_init();  // release of the barrier inits to the cluster
  }
  __syncthreads();
  // the other ranks store into rank 0's shared memory only after this arrival of
  // every thread of rank 0 (its barriers are initialised); rank 0 never waits on it
  if (split > 1) asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  bool failed = false;

  if (warp == kCWarps) {
    // ------------------------------------------------------------ producer --
    if (elect_one_sync()) {
      prefetch_tmap(tmW);
      prefetch_tmap(tmS);
      prefetch_tmap(tmB);
      const uint32_t tx = (uint32_t)geo.R * ((uint32_t)KS / 2u + 2u * geo.sbytes);
      int s = 0, round = 0;
      for (int i = 0; i < nst; ++i) {
        if (i == kXPre) mbar_wait(xready, 0, err, failed);
        if (round > 0) mbar_wait(&empty[s], (round - 1) & 1, err, failed);
        uint8_t* sl = smem + s * geo.slot;
        mbar_arrive_expect_tx(&full[s], tx);
        const int kb = kb0 + i;
        for (int h = 0; h < nbox; ++h) tma_load_2d(sl + h * geo.cb, tmW, &full[s], (kb * KS + h * 256) / 2, r0);
        uint8_t* ss = sl + nbox * geo.cb;
        tma_load_2d(ss, tmS, &full[s], kb * (KS / GROUP), r0);
        tma_load_2d(ss + geo.RG * 16 * geo.sbytes, tmB, &full[s], kb * (KS / GROUP), r0);
        if (++s == geo.nslots) { s = 0; ++round; }
      }
      // no copy may still be writing shared memory when the CTA exits (the waits
      // run, bounded, even after an earlier one expired)
      bool drain_failed = false;
      for (int i = max(0, nst - geo.nslots); i < nst; ++i)
        mbar_wait(&full[i % geo.nslots], (i / geo.nslots) & 1, err, drain_failed);
      // every weight byte of this CTA has landed: warm L2 for the next launch (AffNext)
      if (next.count > 0) {
        const int ncta = next.blk0[next.count] * next.split;
        for (int c = blockIdx.x; c < ncta; c += gridDim.x) {
          const int nrank = c % next.split, nbk = c / next.split;
          int m = 0;
          while (m + 1 < next.count && nbk >= next.blk0[m + 1]) ++m;
          const int nr0 = (int)(((int64_t)next.N[m] * (nbk - next.blk0[m])) / (next.blk0[m + 1] - next.blk0[m]));
          const int k0 = (int)(((int64_t)next.nst * nrank) / next.split);
          const int k1 = (int)(((int64_t)next.nst * (nrank + 1)) / next.split);
          for (int i = k0; i < min(k1, k0 + next.stages); ++i) {
            for (int h = 0; h < next.ks / 256; ++h)
              asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];"
                           :: "l"(&next.tmW[m]), "r"((i * next.ks + h * 256) / 2), "r"(nr0) : "memory");
            asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];"
                         :: "l"(&next.tmS[m]), "r"(i * (next.ks / GROUP)), "r"(nr0) : "memory");
            asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];"
                         :: "l"(&next.tmB[m]), "r"(i * (next.ks / GROUP)), "r"(nr0) : "memory");
          }
        }
      }
    }
    return;
  }

  // ------------------------------------------------------------- consumers --
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // x -> f16 in the decode's pair order (e0,e4)(e1/16,e5/16)(e2,e6)(e3/16,e7/16),
  // one power-of-two pre-scale per scale group (the group's chunks are in
  // neighbouring lanes; the loop's range test is uniform within each group)
  const int tid = threadIdx.x;  // 0 .. 511
  if (tid < 4) zero16[tid] = make_uint4(0, 0, 0, 0);
  for (int c = tid; c < C; c += kCWarps * 32) {
    const unsigned mask = __activemask();
    const uint4* src = reinterpret_cast<const uint4*>(x + (int64_t)kb0 * KS + c * 32);
    uint4 xv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) xv[i] = __ldg(src + i);
    uint32_t mb = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) mb = max(mb, max_mag8(xv[i]));
#pragma unroll
    for (int o = 1; o < kLpg; o <<= 1) mb = max(mb, __shfl_xor_sync(mask, mb, o));
    int sigma = 0;
    if (mb != 0) {
      const int E = (int)(mb >> 7);
      const int e = (E == 0) ? (-133 + (31 - __clz((int)(mb & 0x7Fu)))) : (E - 127);
      sigma = min(14 - e, 127);
    }
    const float xscale = exp2i_f32(sigma);
    float s1 = 0.f, s2 = 0.f;
    uint4* dst = reinterpret_cast<uint4*>(xs + c * 32);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t v[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w};
      float f[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        f[2 * j] = bf16_lo(v[j]) * xscale;
        f[2 * j + 1] = bf16_hi(v[j]) * xscale;
      }
      const uint4 o = make_uint4(f16x2_bits(f[0], f[4]), f16x2_bits(f[1] * 0.0625f, f[5] * 0.0625f),
                                 f16x2_bits(f[2], f[6]), f16x2_bits(f[3] * 0.0625f, f[7] * 0.0625f));
      const __half2* hp = reinterpret_cast<const __half2*>(&o);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 hf = __half22float2(hp[j]);
        s1 += hf.x + hf.y;
        s2 += (hf.x + hf.y) * ((j & 1) ? 16.0f : 1.0f);
      }
      dst[i] = o;
    }
    const float P = exp2i_f32(-sigma);
    if (CF::kPairs) {  // chunk pair (2m, 2m + 1): neighbouring lanes, one scale group
      s1 += __shfl_xor_sync(mask, s1, 1);
      s2 += __shfl_xor_sync(mask, s2, 1);
      if ((c & 1) == 0) cst[c >> 1] = make_float4(P, 1024.f * P * s1, P * s2, 0.f);
    } else {
      cst[c] = make_float4(P, 1024.f * P * s1, P * s2, 0.f);
    }
  }
  asm volatile("bar.sync 1, %0;" :: "n"(kCWarps * 32) : "memory");
  if (tid == 0) mbar_arrive(xready);

  const int jj = warp % IPS, wr = warp / IPS;  // item column, first row group
  const int g = lane >> 2, t = lane & 3;
  // MMA row g holds W row pg = g / 2 + 4 (g % 2) of the 16-row group (and g + 8 row pg + 8):
  // the two rows a quarter-warp reads then sit in different halves of the 128-byte
  // swizzle pattern, so their 16-byte pieces fall in disjoint shared-memory banks
  const int pgr = (g >> 1) | ((g & 1) << 2);
  const bool x_lane = (lane < 20) && (lane % 5 == 0);  // lanes 0, 5, 10, 15 carry B column lane / 5
  const uint32_t zero_addr = smem_u32(zero16);
  const uint32_t xs_addr = smem_u32(xs);
  const uint32_t cst_addr = smem_u32(cst);
  const uint32_t bias_off = (uint32_t)geo.RG * 16u * geo.sbytes;
  float acc[RGW][2];
#pragma unroll
  for (int r = 0; r < RGW; ++r) acc[r][0] = acc[r][1] = 0.f;

  int s = 0, round = 0;
  for (int i = 0; i < nst; ++i) {
    mbar_wait(&full[s], round & 1, err, failed);
    const uint32_t sl = base + s * geo.slot;
    const int cbase = (i * KS + jj * 128) >> 5;  // first chunk of this warp's item column
    // B: x of chunk lane / 5 at lane 5 i, zeros elsewhere
    const uint32_t xp = x_lane ? xs_addr + (uint32_t)(cbase + lane / 5) * 64u : zero_addr;
    const uint4 xa0 = lds128(xp), xa1 = lds128(xp + 16), xa2 = lds128(xp + 32), xa3 = lds128(xp + 48);
    const uint32_t xb[16] = {xa0.x, xa0.y, xa0.z, xa0.w, xa1.x, xa1.y, xa1.z, xa1.w,
                             xa2.x, xa2.y, xa2.z, xa2.w, xa3.x, xa3.y, xa3.z, xa3.w};
    // lanes t < 2 own D columns 2t, 2t + 1 (chunks of the item): their constants
    float4 k0 = make_float4(0.f, 0.f, 0.f, 0.f), k1 = k0;
    if (t < 2) {
      if (CF::kPairs) {
        k0 = lds128f(cst_addr + (uint32_t)((cbase >> 1) + t) * 16u);
      } else {
        k0 = lds128f(cst_addr + (uint32_t)(cbase + 2 * t) * 16u);
        k1 = lds128f(cst_addr + (uint32_t)(cbase + 2 * t + 1) * 16u);
      }
    }
    const int gi0 = (jj * 128 + 2 * t * 32) / GROUP;         // scale group of chunk 2t in the stage
    const int gi1 = (jj * 128 + (2 * t + 1) * 32) / GROUP;   // and of chunk 2t + 1
    const uint32_t box = sl + (uint32_t)(jj >> 1) * geo.cb;
    const int piece = (jj & 1) * 4 + t;  // 16-byte piece (chunk t of the item) of the 128-byte box row
    const uint32_t sbase = sl + (uint32_t)nbox * geo.cb;
#pragma unroll
    for (int r = 0; r < RGW; ++r) {
      const int rg = wr + r * WR;
      if (rg < geo.RG) {  // warp-uniform
        const int rowg = 16 * rg + pgr, rowh = rowg + 8;
        const uint4 qg = lds128(box + (uint32_t)rowg * 128u + (uint32_t)((piece ^ (rowg & 7)) << 4));
        const uint4 qh = lds128(box + (uint32_t)rowh * 128u + (uint32_t)((piece ^ (rowh & 7)) << 4));
        uint32_t pg[16], ph[16];
        decode_word(qg.x, pg);
        decode_word(qg.y, pg + 4);
        decode_word(qg.z, pg + 8);
        decode_word(qg.w, pg + 12);
        decode_word(qh.x, ph);
        decode_word(qh.y, ph + 4);
        decode_word(qh.z, ph + 8);
        decode_word(qh.w, ph + 12);
        float da[4] = {0.f, 0.f, 0.f, 0.f}, db[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int st = 0; st < 8; st += 2) {
          mma_wa(da, pg[2 * st], ph[2 * st], pg[2 * st + 1], ph[2 * st + 1], xb[2 * st], xb[2 * st + 1]);
          mma_wa(db, pg[2 * st + 2], ph[2 * st + 2], pg[2 * st + 3], ph[2 * st + 3], xb[2 * st + 2], xb[2 * st + 3]);
        }
        if (t < 2) {
          // D: c0 = (row g, chunk 2t), c1 = (g, 2t + 1), c2 = (g + 8, 2t), c3 = (g + 8, 2t + 1)
          const uint32_t ag = sbase + (uint32_t)rowg * geo.sbytes, ah = sbase + (uint32_t)rowh * geo.sbytes;
          const float sg0 = lds_bf16(ag + gi0 * 2), bg0 = lds_bf16(ag + bias_off + gi0 * 2);
          const float sh0 = lds_bf16(ah + gi0 * 2), bh0 = lds_bf16(ah + bias_off + gi0 * 2);
          const float d0 = da[0] + db[0], d1 = da[1] + db[1], d2 = da[2] + db[2], d3 = da[3] + db[3];
          if (CF::kPairs) {
            acc[r][0] = fmaf(sg0, fmaf(k0.x, d0 + d1, -k0.y), fmaf(bg0, k0.z, acc[r][0]));
            acc[r][1] = fmaf(sh0, fmaf(k0.x, d2 + d3, -k0.y), fmaf(bh0, k0.z, acc[r][1]));
          } else {
            const float sg1 = lds_bf16(ag + gi1 * 2), bg1 = lds_bf16(ag + bias_off + gi1 * 2);
            const float sh1 = lds_bf16(ah + gi1 * 2), bh1 = lds_bf16(ah + bias_off + gi1 * 2);
            acc[r][0] = fmaf(sg0, fmaf(k0.x, d0, -k0.y), fmaf(bg0, k0.z, acc[r][0]));
            acc[r][0] = fmaf(sg1, fmaf(k1.x, d1, -k1.y), fmaf(bg1, k1.z, acc[r][0]));
            acc[r][1] = fmaf(sh0, fmaf(k0.x, d2, -k0.y), fmaf(bh0, k0.z, acc[r][1]));
            acc[r][1] = fmaf(sh1, fmaf(k1.x, d3, -k1.y), fmaf(bh1, k1.z, acc[r][1]));
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    if (++s == geo.nslots) { s = 0; ++round; }
  }

  // ---- partial row sums: add the two D-holding lanes of a row, then the item columns in order
#pragma unroll
  for (int r = 0; r < RGW; ++r) {
    const int rg = wr + r * WR;
    float vg = acc[r][0] + __shfl_xor_sync(0xffffffffu, acc[r][0], 1);
    float vh = acc[r][1] + __shfl_xor_sync(0xffffffffu, acc[r][1], 1);
    if (rg < geo.RG && t == 0) {
      part[jj * kMaxRows + 16 * rg + pgr] = vg;
      part[jj * kMaxRows + 16 * rg + 8 + pgr] = vh;
    }
  }
  asm volatile("bar.sync 1, %0;" :: "n"(kCWarps * 32) : "memory");
  if (split > 1 && rank > 0) {
    // this rank's row sums into rank 0's shared memory by asynchronous remote
    // stores, which rank 0's barrier counts by bytes
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");  // rank 0 is initialised
    for (int r = tid; r < rows; r += kCWarps * 32) {
      float v = 0.f;
#pragma unroll
      for (int k = 0; k < IPS; ++k) v += part[k * kMaxRows + r];
      asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];"
                   :: "r"(mapa_u32(smem_u32(xpart + rank * kMaxRows + r), 0)), "r"(__float_as_uint(v)),
                      "r"(mapa_u32(smem_u32(pbar), 0)) : "memory");
    }
    return;
  }
  if (split > 1) {
    if (tid == 0) mbar_arrive_expect_tx(pbar, (uint32_t)(split - 1) * (uint32_t)rows * 4u);
    mbar_wait(pbar, 0, err, failed);  // every other rank's row sums have landed
  }
  for (int r = tid; r < rows; r += kCWarps * 32) {
    float v = 0.f;
#pragma unroll
    for (int k = 0; k < IPS; ++k) v += part[k * kMaxRows + r];
    for (int c = 1; c < split; ++c) v += xpart[c * kMaxRows + r];  // in rank order: the same on every run
    mats.y[mi][r0 + r] = (uint16_t)f32_to_bf16_rn(v);
  }
}

// The plan: R rows per row block, the widest stage (IPS item columns) whose
// ring still holds at least three slots, as many slots as fit.  A row block is
// one CTA, or a cluster of 2 or 4 CTAs splitting K when one CTA per SM would
// get fewer than kMinRows rows (the consumers' per-item latency makes short
// blocks slow: 34-row blocks ran at ~2 TB/s; on the affine decode stack a
// threshold of 64 / 96 / 128 / 200 rows gave 54.0 / 57.7 / 58.4 / 58.3 % of HBM).  A group stacks its matrices'
// rows for the block count, then takes the smallest R that gives every matrix
// whole blocks within it.
constexpr int kMinRows = 128;
struct Plan {
  AffGeo geo;
  int ips = 0;
  int split = 1;
  int nb[kMaxGroup] = {0, 0, 0, 0};  // row blocks of each matrix
};

bool plan_geo(int64_t R, int nblk, int64_t K, int split, int group, Plan* p) {
  if (R < 1 || R > kMaxRows) return false;
  for (int ips : {16, 8, 4}) {
    const int KS = 128 * ips;
    if (KS < 8 * group || K % KS != 0 || K / KS < split) continue;
    const int64_t kslice = (K / KS + split - 1) / split * KS;
    if (kslice > kMaxK) continue;
    const uint32_t fixed = 1024u + x_region_bytes((int)kslice, group) + kPartBytes + kXPartBytes + kBarBytes;
    if (fixed >= kSmemBytes) continue;
    AffGeo g;
    g.nblk = nblk;
    g.R = (int)R;
    g.RG = (int)((R + 15) / 16);
    g.cb = (uint32_t)g.RG * 16u * 128u;
    g.sbytes = (uint32_t)(KS / group) * 2u;
    const uint32_t slot = (uint32_t)(KS / 256) * g.cb + 2u * (uint32_t)g.RG * 16u * g.sbytes;
    g.slot = (slot + 1023u) / 1024u * 1024u;
    const uint32_t nslots = std::min<uint32_t>(kMaxSlots, (kSmemBytes - fixed) / g.slot);
    if (nslots < (ips == 4 ? 2u : 3u)) continue;
    g.nslots = (int)nslots;
    p->geo = g;
    p->ips = ips;
    p->split = split;
    return true;
  }
  return false;
}

// Clusters of `split` CTAs of the kernel that can be resident at once (every
// instantiation has the same block and shared memory; cached per device).
int aff_max_clusters(const DevInfo& d, int split) {
  static std::mutex mu;
  static int cache[64][kMaxSplit + 1];
  static bool have[64][kMaxSplit + 1];
  if (d.device < 0 || d.device >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (have[d.device][split]) return cache[d.device][split];
  int n = 0;
  if (cudaFuncSetAttribute(qmv_affine_kernel<64, 16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kSmemBytes) == cudaSuccess) {
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
    if (cudaOccupancyMaxActiveClusters(&n, qmv_affine_kernel<64, 16>, &cfg) != cudaSuccess) n = 0;
  }
  cudaGetLastError();  // a failed query leaves no sticky error behind
  cache[d.device][split] = n;
  have[d.device][split] = true;
  return n;
}

bool plan_split(const DevInfo& d, int count, const int64_t* N, int64_t K, int group, int split, Plan* p) {
  int64_t total = 0;
  for (int i = 0; i < count; ++i) total += N[i];
  const int64_t nblk0 = split == 1 ? std::max<int64_t>(d.sm_count, (total + kMaxRows - 1) / kMaxRows)
                                   : std::min<int64_t>(aff_max_clusters(d, split), d.sm_count / split);
  if (nblk0 < 1) return false;
  if (count == 1) {
    p->nb[0] = (int)std::min<int64_t>(nblk0, N[0]);  // rows per block <= ceil(N / nblk) = R
    return plan_geo((N[0] + nblk0 - 1) / nblk0, p->nb[0], K, split, group, p);
  }
  for (int64_t R = (total + nblk0 - 1) / nblk0; R <= kMaxRows; ++R) {
    int64_t blocks = 0;
    for (int i = 0; i < count; ++i) blocks += (N[i] + R - 1) / R;
    if (blocks <= nblk0) {
      for (int i = 0; i < count; ++i) p->nb[i] = (int)((N[i] + R - 1) / R);
      return plan_geo(R, (int)blocks, K, split, group, p);
    }
  }
  return false;
}

bool plan_affine(const DevInfo& d, int count, const int64_t* N, int64_t K, int group, Plan* p) {
  if (count < 1 || count > kMaxGroup || d.sm_count < 1 || (group != 32 && group != 64 && group != 128))
    return false;
  bool any = false;
  for (int split : {1, 2, 4}) {
    Plan q;
    if (!plan_split(d, count, N, K, group, split, &q)) continue;
    *p = q;
    any = true;
    if (q.geo.R >= kMinRows) break;  // the first split whose blocks are tall enough
  }
  return any;
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

// One matrix's maps for blocks of R rows and stages of KS codes.
bool make_maps(CUtensorMap* tw, CUtensorMap* ts, CUtensorMap* tb, const void* w, const void* scales,
               const void* biases, int64_t N, int64_t K, int group, int R, int KS) {
  const uint64_t groups = (uint64_t)(K / group);
  return make_map(tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, (uint64_t)K / 2, (uint64_t)N, (uint64_t)K / 2, 128,
                  (uint32_t)R, CU_TENSOR_MAP_SWIZZLE_128B) &&
         make_map(ts, CU_TENSOR_MAP_DATA_TYPE_UINT16, scales, groups, (uint64_t)N, groups * 2, (uint32_t)(KS / group),
                  (uint32_t)R, CU_TENSOR_MAP_SWIZZLE_NONE) &&
         make_map(tb, CU_TENSOR_MAP_DATA_TYPE_UINT16, biases, groups, (uint64_t)N, groups * 2, (uint32_t)(KS / group),
                  (uint32_t)R, CU_TENSOR_MAP_SWIZZLE_NONE);
}

constexpr int kPrefetchStages = 3;  // stages of the next launch warmed in L2 (as the FP4 GEMV)

template <int GROUP, int IPS>
cudaError_t launch_group(const DevInfo& d, const Plan& p, const AffGroup& g, const AffNext& nx, const uint16_t* x,
                         int64_t K, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(qmv_affine_kernel<GROUP, IPS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.geo.nblk * p.split));
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
  return cudaLaunchKernelEx(&cfg, qmv_affine_kernel<GROUP, IPS>, g, nx, x, (int)K, p.split, p.geo, d.err);
}

template <int GROUP>
cudaError_t launch_ips(const DevInfo& d, const Plan& p, const AffGroup& g, const AffNext& nx, const uint16_t* x,
                       int64_t K, cudaStream_t s) {
  if (p.ips == 16) return launch_group<GROUP, 16>(d, p, g, nx, x, K, s);
  if (p.ips == 8) return launch_group<GROUP, 8>(d, p, g, nx, x, K, s);
  if (GROUP <= 64 && p.ips == 4) return launch_group<GROUP, (GROUP <= 64 ? 4 : 8)>(d, p, g, nx, x, K, s);
  return cudaErrorInvalidValue;
}

}  // namespace

bool qmv_affine_supported(const DevInfo& d, int64_t N, int64_t K, int group) {
  Plan p;
  return plan_affine(d, 1, &N, K, group, &p);
}

bool qmv_affine_group_supported(const DevInfo& d, int count, const int64_t* N, int64_t K, int group) {
  Plan p;
  return plan_affine(d, count, N, K, group, &p);
}

cudaError_t launch_qmv_affine_group(const DevInfo& d, const uint16_t* x, int count, const uint32_t* const* w,
                                    const uint16_t* const* scales, const uint16_t* const* biases, const int64_t* N,
                                    int64_t K, int group, uint16_t* const* y, const GemvGroupDesc* nextd,
                                    cudaStream_t s) {
  Plan p;
  if (!plan_affine(d, count, N, K, group, &p)) return cudaErrorInvalidValue;
  AffGroup g;
  memset(&g, 0, sizeof(g));
  g.count = count;
  for (int i = 0; i < count; ++i) {
    if (!make_maps(&g.tmW[i], &g.tmS[i], &g.tmB[i], w[i], scales[i], biases[i], N[i], K, group, p.geo.R,
                   128 * p.ips))
      return cudaErrorInvalidValue;
    g.y[i] = y[i];
    g.N[i] = (int)N[i];
    g.blk0[i + 1] = g.blk0[i] + p.nb[i];
  }
  // the next launch as it will be planned (a hint: dropped if it has no plan)
  AffNext nx;
  memset(&nx, 0, sizeof(nx));
  if (nextd && nextd->count >= 1 && nextd->count <= kMaxGroup) {
    Plan np;
    bool ok = plan_affine(d, nextd->count, nextd->N, nextd->K, group, &np);
    for (int i = 0; ok && i < nextd->count; ++i) {
      ok = nextd->biases[i] != nullptr &&
           make_maps(&nx.tmW[i], &nx.tmS[i], &nx.tmB[i], nextd->w[i], nextd->scales[i], nextd->biases[i],
                     nextd->N[i], nextd->K, group, np.geo.R, 128 * np.ips);
      nx.N[i] = (int)nextd->N[i];
      nx.blk0[i + 1] = nx.blk0[i] + np.nb[i];
    }
    if (ok) {
      nx.count = nextd->count;
      nx.ks = 128 * np.ips;
      nx.nst = (int)(nextd->K / nx.ks);
      nx.split = np.split;
      nx.stages = kPrefetchStages;
    } else {
      memset(&nx, 0, sizeof(nx));
    }
  }
  if (group == 32) return launch_ips<32>(d, p, g, nx, x, K, s);
  if (group == 64) return launch_ips<64>(d, p, g, nx, x, K, s);
  if (group == 128) return launch_ips<128>(d, p, g, nx, x, K, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_qmv_affine(const DevInfo& d, const uint16_t* x, const uint32_t* w, const uint16_t* scales,
                              const uint16_t* biases, int64_t N, int64_t K, int group, uint16_t* y,
                              cudaStream_t s) {
  return launch_qmv_affine_group(d, x, 1, &w, &scales, &biases, &N, K, group, &y, nullptr, s);
}

}  // namespace fp4
