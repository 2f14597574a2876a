// qmv_affine.cu -- affine 4-bit decode GEMV (group 32 / 64 / 128, bf16 scale
// and bias) fed by a TMA shared-memory ring.
//
// Pages: "epic: NVIDIA Volta (sm_70) inference acceleration program #1536"
// (Baseline: the decode step streams affine 4-bit group-64 weights at 7.7 % of
// the V100's bandwidth, ALU-bound; Diagnosis 3: the accumulator type -- fp32
// here), "mlx 0.30.7.3 -> 0.30.7.6" quantized.cpp (affine w = q * scale + bias).
//
// The weight stream is the whole cost, so the kernel is built to retire ~27
// weights per SM clock with few instructions each:
//   * warp 16 (one thread) streams W by TMA: per stage of KS codes (KS = 512 for
//     groups of 32 and 64, 1024 for 128) KS / 256 boxes of R rows x 128 bytes
//     (128-byte swizzle) plus one box of R rows of scales and one of biases,
//     into a ring of slots.  The first kXPre stages go out before the previous
//     kernel has finished (programmatic dependent launch: no kernel of this
//     library writes weights and releases its dependents early); later ones wait
//     until x has been staged, whose loads would otherwise queue behind them;
//   * warps 0-15 decode and multiply on the tensor cores with mma.sync
//     m16n8k16 (f16 inputs, fp32 accumulation).  A code byte pair becomes an
//     f16 pair with one LOP3 per pair: (w & 0x000F000F) | 0x64006400 is
//     f16(1024 + q) for nibbles 0 and 4, (w & 0x00F000F0) | 0x64006400 is
//     f16(1024 + 16 q) for nibbles 1 and 5, and the same on w >> 8 for nibbles
//     2, 6 and 3, 7: five instructions per eight codes.  x is staged as f16 in
//     that pair order with the nibble-1/3 elements divided by 16, so every
//     product is (1024 + c q) (x / c) = 1024 x / c + q x and the sum over a
//     32-code chunk is D = 1024 X' + sum q x with X' the sum of the staged
//     values;
//   * fragment plan (one warp, one item = 16 weight rows x 128 codes): lane
//     (g, t) = (lane / 4, lane % 4) reads the 32 codes of chunk t of rows g and
//     g + 8; A is zero but for row i at lane 5 i, which holds x at chunk i's
//     positions, so D[i, n] is chunk i's partial dot product for row n and
//     every D element lies inside one scale group: y += 2^-sigma (s (D - 1024 X')
//     + b X), X the chunk's sum of x (per-chunk power-of-two pre-scale sigma
//     keeps every bf16 x exact in f16 down to 2^-24 of the chunk's max);
//   * a CTA owns R <= 256 rows (row groups of 16); warps split as WK warps per
//     row group, each taking every WK-th item of its row group, so a warp's
//     accumulators stay in registers; the partial row sums meet in shared
//     memory and are added in warp order (deterministic).
// Every mbarrier wait is bounded (an expired wait records FP4_ERR_TIMEOUT).
#include <algorithm>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "launch.h"

namespace fp4 {

namespace {

constexpr int kCWarps = 16;                   // consumer warps
constexpr int kThreads = (kCWarps + 1) * 32;  // + the TMA producer warp
constexpr int kMaxK = 32768;                  // x is staged whole in shared memory
constexpr int kMaxRows = 256;                 // rows per CTA (TMA box height)
constexpr int kMaxSlots = 24;
constexpr int kXPre = 4;                      // stages issued before x has been staged
constexpr uint32_t kSmemBytes = 227u * 1024u;
constexpr uint32_t kBarBytes = 512;
constexpr uint32_t kPartBytes = kCWarps * 16 * 4;
static_assert(2 * kMaxSlots + 2 <= kBarBytes / 8, "barrier area");

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}

__device__ __forceinline__ uint32_t lds16(uint32_t a) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
  return v;
}

__device__ __forceinline__ uint32_t f16x2_bits(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// one 32-bit word of eight codes -> the four f16 pairs of the plan above
__device__ __forceinline__ void decode_word(uint32_t w, uint32_t& p0, uint32_t& p1, uint32_t& p2, uint32_t& p3) {
  const uint32_t w8 = w >> 8;
  p0 = (w & 0x000F000Fu) | 0x64006400u;   // 1024 + q0, 1024 + q4
  p1 = (w & 0x00F000F0u) | 0x64006400u;   // 1024 + 16 q1, 1024 + 16 q5
  p2 = (w8 & 0x000F000Fu) | 0x64006400u;  // 1024 + q2, 1024 + q6
  p3 = (w8 & 0x00F000F0u) | 0x64006400u;  // 1024 + 16 q3, 1024 + 16 q7
}

struct AffGeo {
  int nblk = 0;        // CTAs (row blocks)
  int R = 0;           // rows per CTA at most (blocks own R or R - 1)
  int RG = 0;          // 16-row groups per CTA
  int WK = 0;          // warps per row group
  int KS = 0;          // codes per stage
  int nslots = 0;      // ring slots
  uint32_t cb = 0;     // bytes of one code box region (RG * 16 rows * 128 B)
  uint32_t sbytes = 0; // scale (and bias) bytes per row per stage
  uint32_t slot = 0;   // bytes per slot
};

// Shared memory (from a 1024-aligned base): [ring | x f16 (K) | X' (C) | X (C) |
// 2^-sigma (C) | 64 zero bytes | partial sums | barriers], C = K / 32.
__host__ __device__ inline uint32_t x_region_bytes(int K) { return (uint32_t)K * 2u + 3u * (uint32_t)(K / 32) * 4u + 64u; }

template <int GROUP>
__global__ void __launch_bounds__(kThreads, 1) qmv_affine_kernel(
    const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmS,
    const __grid_constant__ CUtensorMap tmB, const uint16_t* __restrict__ x, int N, int K, AffGeo geo,
    uint16_t* __restrict__ y, unsigned* __restrict__ err) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const int C = K >> 5;
  const uint32_t ring_bytes = (uint32_t)geo.nslots * geo.slot;
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem + ring_bytes);
  float* xs1 = reinterpret_cast<float*>(smem + ring_bytes + (uint32_t)K * 2u);  // X': sum of staged values
  float* xs2 = xs1 + C;                                                          // X: sum of pre-scaled x
  float* xinv = xs2 + C;                                                         // 2^-sigma
  uint4* zero16 = reinterpret_cast<uint4*>(xinv + C);
  float* part = reinterpret_cast<float*>(smem + ring_bytes + x_region_bytes(K));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + ring_bytes + x_region_bytes(K) + kPartBytes);
  uint64_t* empty = full + kMaxSlots;
  uint64_t* xready = empty + kMaxSlots;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nblk = gridDim.x;
  const int r0 = (int)(((int64_t)N * blockIdx.x) / nblk);
  const int rows = (int)(((int64_t)N * (blockIdx.x + 1)) / nblk) - r0;  // <= R
  const int nst = K / geo.KS;
  const int nbox = geo.KS / 256;
  const int ips = geo.KS / 128;  // items (128 codes) per row group per stage

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) {
    for (int s = 0; s < geo.nslots; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kCWarps);
    }
    mbar_init(xready, 1);
    fence_barrier_init();
  }
  __syncthreads();
  bool failed = false;

  if (warp == kCWarps) {
    // ------------------------------------------------------------ producer --
    if (elect_one_sync()) {
      prefetch_tmap(&tmW);
      prefetch_tmap(&tmS);
      prefetch_tmap(&tmB);
      const uint32_t tx = (uint32_t)geo.R * ((uint32_t)geo.KS / 2u + 2u * geo.sbytes);
      int s = 0, round = 0;
      for (int i = 0; i < nst; ++i) {
        if (i == kXPre) mbar_wait(xready, 0, err, failed);
        if (round > 0) mbar_wait(&empty[s], (round - 1) & 1, err, failed);
        uint8_t* sl = smem + s * geo.slot;
        mbar_arrive_expect_tx(&full[s], tx);
        for (int h = 0; h < nbox; ++h) tma_load_2d(sl + h * geo.cb, &tmW, &full[s], (i * geo.KS + h * 256) / 2, r0);
        uint8_t* ss = sl + nbox * geo.cb;
        tma_load_2d(ss, &tmS, &full[s], i * (geo.KS / GROUP), r0);
        tma_load_2d(ss + geo.RG * 16 * geo.sbytes, &tmB, &full[s], i * (geo.KS / GROUP), r0);
        if (++s == geo.nslots) { s = 0; ++round; }
      }
      // no copy may still be writing shared memory when the CTA exits
      for (int i = max(0, nst - geo.nslots); i < nst; ++i)
        mbar_wait(&full[i % geo.nslots], (i / geo.nslots) & 1, err, failed);
    }
    return;
  }

  // ------------------------------------------------------------- consumers --
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // x -> f16 in the decode's pair order (e0,e4)(e1/16,e5/16)(e2,e6)(e3/16,e7/16),
  // one power-of-two pre-scale per 32-element chunk: max|x| 2^sigma in [2^14, 2^15).
  const int tid = threadIdx.x;  // 0 .. 511
  if (tid < 4) zero16[tid] = make_uint4(0, 0, 0, 0);
  for (int c = tid; c < C; c += kCWarps * 32) {
    const uint4* src = reinterpret_cast<const uint4*>(x + c * 32);
    uint4 xv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) xv[i] = __ldg(src + i);
    uint32_t mb = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) mb = max(mb, max_mag8(xv[i]));
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
        const float cmul = (j & 1) ? 16.0f : 1.0f;
        s1 += hf.x + hf.y;
        s2 += (hf.x + hf.y) * cmul;
      }
      dst[i] = o;
    }
    xs1[c] = s1;
    xs2[c] = s2;
    xinv[c] = exp2i_f32(-sigma);
  }
  asm volatile("bar.sync 1, %0;" :: "n"(kCWarps * 32) : "memory");
  if (tid == 0) mbar_arrive(xready);

  // warp -> (row group rg, k-lane wk); warps past RG * WK only keep the barrier count
  const int rg = warp / geo.WK, wk = warp % geo.WK;
  const bool active = rg < geo.RG;
  const int g = lane >> 2, t = lane & 3;
  const bool x_lane = (lane < 20) && (lane % 5 == 0);  // lanes 0, 5, 10, 15 carry A row lane / 5
  const uint32_t zero_addr = smem_u32(zero16);
  const uint32_t xs_addr = smem_u32(xs);
  const int src0 = 8 * t + g, src1 = src0 + 4;  // lanes that read rows 2t, 2t + 1 of the D chunk g
  const bool half1 = active && (16 * rg + 8 < rows);
  float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};

  int s = 0, round = 0;
  for (int i = 0; i < nst; ++i) {
    mbar_wait(&full[s], round & 1, err, failed);
    const uint32_t sl = base + s * geo.slot;
    if (active) {
      for (int j = 0; j < ips; ++j) {
        if (((i * ips + j) % geo.WK) != wk) continue;
        const int cbase = (i * geo.KS + j * 128) >> 5;  // first chunk of the item
        // x fragments of chunk lane / 5 (A row lane / 5), zeros elsewhere
        const uint32_t xp = x_lane ? xs_addr + (uint32_t)(cbase + lane / 5) * 64u : zero_addr;
        const uint4 xa0 = lds128(xp), xa1 = lds128(xp + 16), xa2 = lds128(xp + 32), xa3 = lds128(xp + 48);
        const int cd = cbase + g;  // chunk of this lane's D elements (lanes 0..15)
        const float xi = lane < 16 ? xinv[cd] : 0.f;
        const float X1 = lane < 16 ? xs1[cd] : 0.f;
        const float X2 = lane < 16 ? xs2[cd] : 0.f;
        const uint32_t box = sl + (uint32_t)(j >> 1) * geo.cb;
        const int piece = (j & 1) * 4 + t;  // 16-byte piece of the 128-byte box row
        const int gi = (j * 128 + t * 32) / GROUP;  // scale group of this lane's chunk in the stage
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (h == 1 && !half1) break;  // the second 8-row half lies past the block (warp-uniform)
          const int row = 16 * rg + 8 * h + g;
          const uint4 q = lds128(box + (uint32_t)row * 128u + (uint32_t)((piece ^ (row & 7)) << 4));
          // this lane's (row, group) scale and bias, packed, for the D holders
          const uint32_t sa = sl + (uint32_t)nbox * geo.cb + (uint32_t)row * geo.sbytes + (uint32_t)gi * 2u;
          const uint32_t sv = lds16(sa) | (lds16(sa + (uint32_t)geo.RG * 16u * geo.sbytes) << 16);
          uint32_t bq[16];
          decode_word(q.x, bq[0], bq[1], bq[2], bq[3]);
          decode_word(q.y, bq[4], bq[5], bq[6], bq[7]);
          decode_word(q.z, bq[8], bq[9], bq[10], bq[11]);
          decode_word(q.w, bq[12], bq[13], bq[14], bq[15]);
          float da[4] = {0.f, 0.f, 0.f, 0.f}, db[4] = {0.f, 0.f, 0.f, 0.f};
          mma_f16(da, xa0.x, xa0.y, bq[0], bq[1]);
          mma_f16(db, xa2.x, xa2.y, bq[8], bq[9]);
          mma_f16(da, xa0.z, xa0.w, bq[2], bq[3]);
          mma_f16(db, xa2.z, xa2.w, bq[10], bq[11]);
          mma_f16(da, xa1.x, xa1.y, bq[4], bq[5]);
          mma_f16(db, xa3.x, xa3.y, bq[12], bq[13]);
          mma_f16(da, xa1.z, xa1.w, bq[6], bq[7]);
          mma_f16(db, xa3.z, xa3.w, bq[14], bq[15]);
          const uint32_t s0 = __shfl_sync(0xffffffffu, sv, src0);
          const uint32_t s1v = __shfl_sync(0xffffffffu, sv, src1);
          // D = 1024 X' + sum q x (pre-scaled)  ->  s (D - 1024 X') + b X
          acc[h][0] = fmaf(fmaf(bf16_lo(s0), (da[0] + db[0]) - 1024.f * X1, bf16_hi(s0) * X2), xi, acc[h][0]);
          acc[h][1] = fmaf(fmaf(bf16_lo(s1v), (da[1] + db[1]) - 1024.f * X1, bf16_hi(s1v) * X2), xi, acc[h][1]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    if (++s == geo.nslots) { s = 0; ++round; }
  }

  // ---- partial row sums: add the four chunk lanes, then across the WK warps in order
  if (active) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float v0 = acc[h][0] + __shfl_xor_sync(0xffffffffu, acc[h][0], 4);
      float v1 = acc[h][1] + __shfl_xor_sync(0xffffffffu, acc[h][1], 4);
      v0 += __shfl_xor_sync(0xffffffffu, v0, 8);
      v1 += __shfl_xor_sync(0xffffffffu, v1, 8);
      if (lane < 4) {
        part[warp * 16 + 8 * h + 2 * lane] = v0;
        part[warp * 16 + 8 * h + 2 * lane + 1] = v1;
      }
    }
  }
  asm volatile("bar.sync 1, %0;" :: "n"(kCWarps * 32) : "memory");
  for (int r = tid; r < rows; r += kCWarps * 32) {
    const int rgr = r >> 4;
    float v = 0.f;
    for (int k = 0; k < geo.WK; ++k) v += part[(rgr * geo.WK + k) * 16 + (r & 15)];
    y[r0 + r] = (uint16_t)f32_to_bf16_rn(v);
  }
}

// The plan: one CTA per SM (more when N > 256 per SM), R rows per CTA, WK
// warps per 16-row group, KS codes per stage, as many ring slots as fit.
bool plan_affine(const DevInfo& d, int64_t N, int64_t K, int group, AffGeo* g) {
  if (K > kMaxK || d.sm_count < 1) return false;
  const int KS = std::max(512, 8 * group);
  if (K % KS != 0) return false;
  const int64_t nblk = std::max<int64_t>(d.sm_count, (N + kMaxRows - 1) / kMaxRows);
  const int64_t R = (N + nblk - 1) / nblk;
  if (R < 1 || R > kMaxRows) return false;
  g->nblk = (int)std::min<int64_t>(nblk, N);  // rows per block <= ceil(N / nblk) = R
  g->R = (int)R;
  g->RG = (int)((R + 15) / 16);
  g->WK = std::max(1, kCWarps / g->RG);
  g->KS = KS;
  g->cb = (uint32_t)g->RG * 16u * 128u;
  g->sbytes = (uint32_t)(KS / group) * 2u;
  const uint32_t slot = (uint32_t)(KS / 256) * g->cb + 2u * (uint32_t)g->RG * 16u * g->sbytes;
  g->slot = (slot + 1023u) / 1024u * 1024u;
  const uint32_t fixed = 1024u + x_region_bytes((int)K) + kPartBytes + kBarBytes;
  if (fixed >= kSmemBytes) return false;
  const uint32_t nslots = std::min<uint32_t>(kMaxSlots, (kSmemBytes - fixed) / g->slot);
  if (nslots < 2) return false;
  g->nslots = (int)nslots;
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
      !make_map(&ts, CU_TENSOR_MAP_DATA_TYPE_UINT16, scales, groups, (uint64_t)N, groups * 2,
                (uint32_t)(geo.KS / GROUP), (uint32_t)geo.R, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !make_map(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT16, biases, groups, (uint64_t)N, groups * 2,
                (uint32_t)(geo.KS / GROUP), (uint32_t)geo.R, CU_TENSOR_MAP_SWIZZLE_NONE))
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
