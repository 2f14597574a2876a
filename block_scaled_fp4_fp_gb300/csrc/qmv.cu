// qmv.cu -- M = 1 decode GEMV against 4-bit weights (affine, NVFP4, MXFP4).
//
// Pages: "epic: NVIDIA Volta (sm_70) inference acceleration program #1536"
// (Baseline: the decode step is the qmv weight stream, measured ALU-bound at
// 7.7 % of HBM; Diagnosis 3: the accumulator type -- here always fp32),
// "mlx 0.30.7.3 -> 0.30.7.6" qqmm.cpp (the M = 1 route through fp_qmv; W
// stored [N, K]).
//
// Why this shape: at ~7 TB/s a GB300 must retire ~2 weights per SM clock per
// SM sub-partition, so the per-weight instruction count decides whether the
// kernel is bandwidth- or issue-bound.  Decoding to fp32 and using FFMA costs
// 2.5+ instructions per weight.  Here the dot products run on the tensor cores
// (mma.sync m16n8k16, f16 inputs, fp32 accumulation): the hardware converter
// turns one byte of two e2m1 codes into exactly the f16x2 register the B
// fragment wants (affine codes use the 0x6400 magic: f16(1024 + q)), so the
// decode is half an instruction per weight and one MMA covers 128 weights.
//
// Fragment plan for one warp and one "item" (16 weight rows x 128 codes, two
// n8 halves sharing one set of x fragments):
//   lane (g, t) = (lane/4, lane%4) loads 16 bytes (32 codes) of rows g and g+8, chunk t;
//   MMA step s (0..7) feeds that lane's codes 4s..4s+3 as its B fragment
//   (column n = g, k positions {2t, 2t+1, 2t+8, 2t+9});
//   A is zero except row i at lanes 5i (i = 0..3), which hold x at the same
//   code positions of chunk i -- so D[i, n] is the partial dot product of the
//   codes lane (n, i) holds, and every D element sees codes of ONE block-scale
//   group: the scale (E4M3 / E8M0 / affine s, b) is applied in fp32 on D.
// x enters as f16 after an exact power-of-two pre-scale chosen per 32-element
// chunk from the chunk's max|x| (max*2^sigma in [2^14, 2^15)); bf16 values are
// exact in f16 there, and only values below max*2^-28 lose bits.  Each D
// element holds one chunk, so 2^-sigma is applied together with the block
// scale; the NVFP4 weight global scale is applied to the finished row sums.
//
// Work split: one persistent CTA per SM, each owning a contiguous row range
// balanced to +-1 row; its (16-row group x 256-code) pipeline stages are split
// into contiguous ranges over 16 warps; every warp streams its weights through
// its own cp.async ring (each lane re-reads only the 16-byte pieces it copied,
// so no barrier is needed), and per-row partial sums meet in shared memory.
#include <algorithm>
#include <cuda_fp16.h>

#include "common.cuh"
#include "launch.h"

namespace fp4 {

namespace {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kB = 2;    // items (16 rows x 128 codes) per pipeline stage
constexpr int kNST = 3;  // stages in each warp's cp.async ring (two in flight while one is consumed)
constexpr int kItemBytes = 2 * 32 * 16;          // two 16-byte loads per lane
constexpr int kRingBytes = kNST * kB * kItemBytes;  // per warp

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}

// four bytes of e2m1 code pairs -> four f16x2 registers (byte j -> h[j], low code in the low half)
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t& h0, uint32_t& h1, uint32_t& h2,
                                                  uint32_t& h3) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3) : "r"(w));
}

// two E4M3 bytes (low byte -> low half) -> f16x2, exact
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t v) {
  uint32_t h;
  const uint16_t b = (uint16_t)(v & 0xFFFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(b));
  return h;
}

__device__ __forceinline__ uint32_t f16x2_bits(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" :: "r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}

__device__ __forceinline__ void mma_f16_first(float (&d)[4], uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%10, %10, %10, %10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1), "f"(0.f));
}

// MODE: 0 affine (group 32/64/128), 1 MXFP4 (group 32), 2 NVFP4 (group 16).
// QX (FP4 modes): x is first replaced by fp_dequantize(fp_quantize(x, gs_x)).
template <int MODE, bool QX>
__global__ void __launch_bounds__(kThreads, 1) qmv_kernel(const uint16_t* __restrict__ x,
                                                           const float* __restrict__ gs_x,
                                                           const uint32_t* __restrict__ w,
                                                           const void* __restrict__ scales_v,
                                                           const uint16_t* __restrict__ biases,
                                                           const float* __restrict__ gs_w, int N, int K,
                                                           int group, uint16_t* __restrict__ y) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int C = K >> 5;                    // 32-code chunks per row
  const int QC = (C + 3) >> 2;             // items (4 chunks) per row
  const int SPR = (QC + kB - 1) / kB;      // pipeline stages per 16-row group
  const int r0 = (int)(((int64_t)N * blockIdx.x) / gridDim.x);
  const int r1 = (int)(((int64_t)N * (blockIdx.x + 1)) / gridDim.x);
  const int RG = (r1 - r0 + 15) >> 4;
  // shared memory: [ring: kWarps x kRingBytes][x f16: K][64 zero bytes][xsum: C floats]
  //                [xinv: C floats, 2^-sigma of each chunk][ypart: RG*16 floats]
  const uint32_t ring = smem_u32(smem) + (threadIdx.x >> 5) * kRingBytes;
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem + kWarps * kRingBytes);
  uint4* zero16 = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(xs) + (size_t)K * 2);
  float* xsum = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(zero16) + 64);
  float* xinv = xsum + C;
  float* ypart = xinv + C;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int words = K >> 3;
  constexpr int SB = (MODE == 2) ? 2 : 1;  // scale bytes per chunk (NVFP4 / MXFP4)

  // ---- this warp's stages: contiguous, each inside one 16-row group
  const int S = RG * SPR;
  const int sb = (int)(((int64_t)S * warp) / kWarps), se = (int)(((int64_t)S * (warp + 1)) / kWarps);

  // issue cursor (stage -> row group rg_i, stage-in-row qs_i) and this lane's pointers for rows g, g+8
  int rg_i = sb / SPR, qs_i = sb - (sb / SPR) * SPR;
  const uint32_t* pw[2] = {nullptr, nullptr};
  const uint8_t* ps[2] = {nullptr, nullptr};
  const uint16_t* pa[2] = {nullptr, nullptr};
  const uint16_t* pb[2] = {nullptr, nullptr};
  bool row_ok[2] = {false, false};
  auto seek = [&]() {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int row = r0 + rg_i * 16 + 8 * h + g;
      row_ok[h] = row < r1;
      const int rr = row_ok[h] ? row : r0;
      const int c = qs_i * kB * 4 + t;
      pw[h] = w + (int64_t)rr * words + c * 4;
      if (MODE != 0) ps[h] = reinterpret_cast<const uint8_t*>(scales_v) + (int64_t)rr * (C * SB) + c * SB;
      else {
        pa[h] = reinterpret_cast<const uint16_t*>(scales_v) + (int64_t)rr * (K / group);
        pb[h] = biases + (int64_t)rr * (K / group);
      }
    }
  };
  uint32_t sc[kNST][kB][2];
  auto issue = [&](int j, uint32_t slot, uint32_t (&scs)[kB][2]) {
    const bool live = (sb + j) < se;
    const int c0 = qs_i * kB * 4 + t;
#pragma unroll
    for (int u = 0; u < kB; ++u) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const bool valid = live && row_ok[h] && (c0 + 4 * u) < C;
        cp_async16(slot + u * kItemBytes + h * 512 + lane * 16, valid ? (const void*)(pw[h] + 16 * u) : (const void*)w,
                   valid ? 16u : 0u);
        uint32_t sv = 0;
        if (valid) {
          if (MODE == 2) sv = __ldg(reinterpret_cast<const uint16_t*>(ps[h] + 8 * u));
          else if (MODE == 1) sv = __ldg(ps[h] + 4 * u);
          else {
            const int gi = ((c0 + 4 * u) << 5) / group;
            sv = (uint32_t)__ldg(pa[h] + gi) | ((uint32_t)__ldg(pb[h] + gi) << 16);
          }
        }
        scs[u][h] = sv;
      }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    if (live) {
      if (++qs_i == SPR) { qs_i = 0; ++rg_i; seek(); }
      else {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          pw[h] += kB * 16;
          if (MODE != 0) ps[h] += kB * 4 * SB;
        }
      }
    }
  };
  // Programmatic dependent launch: let the next kernel in the stream start
  // launching now, and stream this kernel's weights (which no earlier kernel
  // writes) before waiting for the previous grid -- x may be its output.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  seek();
#pragma unroll
  for (int p = 0; p < kNST - 1; ++p) issue(p, ring + p * kB * kItemBytes, sc[p]);
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // ---- x -> f16 in shared memory, one power-of-two pre-scale per 32-element
  // chunk: max|x|*2^sigma in [2^14, 2^15), so every bf16 value of the chunk
  // above max*2^-28 is exact in f16.  Each D element of the main loop holds
  // one chunk's partial sum, so 2^-sigma is applied with the block scale.
  for (int i = tid; i < RG * 16; i += kThreads) ypart[i] = 0.f;
  if (tid < 4) zero16[tid] = make_uint4(0, 0, 0, 0);
  for (int c = tid; c < C; c += kThreads) {
    const uint4* src = reinterpret_cast<const uint4*>(x + c * 32);
    uint4 xv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) xv[i] = __ldg(src + i);
    if (QX) {  // this chunk is two NVFP4 blocks or one MXFP4 block
      const float gsx = (MODE == 2 && gs_x) ? __ldg(gs_x) : 1.0f;
#pragma unroll
      for (int b = 0; b < (MODE == 2 ? 2 : 1); ++b) {
        constexpr int NB = (MODE == 2) ? 2 : 4;
        uint32_t mb = 0;
#pragma unroll
        for (int i = 0; i < NB; ++i) mb = max(mb, max_mag8(xv[b * NB + i]));
        float mul, sval;
        uint32_t sbyte;
        block_scale_rule<(MODE == 2 ? 2 : 1)>(mb, gsx, mul, sbyte, sval);
#pragma unroll
        for (int i = 0; i < NB; ++i) xv[b * NB + i] = quant_dequant8(xv[b * NB + i], mul, sval, gsx);
      }
    }
    uint32_t m2 = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      m2 = __vmaxu2(m2, xv[i].x & 0x7FFF7FFFu);
      m2 = __vmaxu2(m2, xv[i].y & 0x7FFF7FFFu);
      m2 = __vmaxu2(m2, xv[i].z & 0x7FFF7FFFu);
      m2 = __vmaxu2(m2, xv[i].w & 0x7FFF7FFFu);
    }
    const uint32_t mb = max(m2 & 0xFFFFu, m2 >> 16);
    int sigma = 0;
    if (mb != 0) {
      const int E = (int)(mb >> 7);
      const int e = (E == 0) ? (-133 + (31 - __clz((int)(mb & 0x7Fu)))) : (E - 127);
      sigma = min(14 - e, 127);
    }
    const float xscale = exp2i_f32(sigma);
    float xsum_c = 0.f;
    uint4* dst = reinterpret_cast<uint4*>(xs + c * 32);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float f0 = bf16_lo(xv[i].x) * xscale, f1 = bf16_hi(xv[i].x) * xscale, f2 = bf16_lo(xv[i].y) * xscale,
                  f3 = bf16_hi(xv[i].y) * xscale, f4 = bf16_lo(xv[i].z) * xscale, f5 = bf16_hi(xv[i].z) * xscale,
                  f6 = bf16_lo(xv[i].w) * xscale, f7 = bf16_hi(xv[i].w) * xscale;
      uint4 o;
      if (MODE == 0) {  // pair order of the 0x6400 affine decode: (e0,e4)(e1,e5)(e2,e6)(e3,e7)
        o = make_uint4(f16x2_bits(f0, f4), f16x2_bits(f1, f5), f16x2_bits(f2, f6), f16x2_bits(f3, f7));
        const __half2* hp = reinterpret_cast<const __half2*>(&o);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 f = __half22float2(hp[j]);
          xsum_c += f.x + f.y;
        }
      } else {
        o = make_uint4(f16x2_bits(f0, f1), f16x2_bits(f2, f3), f16x2_bits(f4, f5), f16x2_bits(f6, f7));
      }
      dst[i] = o;
    }
    if (MODE == 0) xsum[c] = xsum_c;
    xinv[c] = exp2i_f32(-sigma);
  }
  __syncthreads();

  // ---- main loop over pipeline stages
  const bool x_lane = (lane < 20) && (lane % 5 == 0);  // lanes 0, 5, 10, 15 carry A row lane/5
  const uint32_t x_base = smem_u32(xs) + (lane / 5) * 64;
  const uint32_t zero_addr = smem_u32(zero16);
  const int src0 = 8 * (lane & 3) + (lane >> 2), src1 = src0 + 4;
  int rg_c = sb / SPR, qs_c = sb - (sb / SPR) * SPR;  // compute cursor
  int rg_acc = rg_c;
  float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};  // [row half][even/odd row of the lane's pair]
  auto flush = [&]() {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float v0 = acc[h][0] + __shfl_xor_sync(0xffffffffu, acc[h][0], 4);
      float v1 = acc[h][1] + __shfl_xor_sync(0xffffffffu, acc[h][1], 4);
      v0 += __shfl_xor_sync(0xffffffffu, v0, 8);
      v1 += __shfl_xor_sync(0xffffffffu, v1, 8);
      if (lane < 4) {
        atomicAdd(&ypart[rg_acc * 16 + 8 * h + 2 * lane], v0);
        atomicAdd(&ypart[rg_acc * 16 + 8 * h + 2 * lane + 1], v1);
      }
    }
  };

  const int nst = se - sb;
  for (int j0 = 0; j0 < nst; j0 += kNST) {
#pragma unroll
    for (int ss = 0; ss < kNST; ++ss) {
      const int j = j0 + ss;
      if (j >= nst) break;
      const int nslot = (ss + kNST - 1) % kNST;
      issue(j + kNST - 1, ring + nslot * kB * kItemBytes, sc[nslot]);
      asm volatile("cp.async.wait_group %0;" :: "n"(kNST - 1) : "memory");
      if (rg_c != rg_acc) {
        flush();
        rg_acc = rg_c;
        acc[0][0] = acc[0][1] = acc[1][0] = acc[1][1] = 0.f;
      }
      const uint32_t slot = ring + ss * kB * kItemBytes;
      const int cbase = qs_c * kB * 4;  // first chunk of this stage
      const bool half1_live = r0 + rg_c * 16 + 8 < r1;
#pragma unroll
      for (int u = 0; u < kB; ++u) {
        const int ci = cbase + 4 * u + (lane / 5);
        const uint32_t xp = (x_lane && ci < C) ? x_base + (cbase + 4 * u) * 64 : zero_addr;
        const uint4 xa0 = lds128(xp), xa1 = lds128(xp + 16), xa2 = lds128(xp + 32), xa3 = lds128(xp + 48);
        const int cd = cbase + 4 * u + (lane >> 2);  // chunk of this lane's D elements
        const bool cd_ok = lane < 16 && cd < C;
        const float xi = cd_ok ? xinv[cd] : 0.f;
        const float X = (MODE == 0 && cd_ok) ? xsum[cd] : 0.f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (h == 1 && !half1_live) break;  // all rows of the second 8-row half lie past the range
          const uint4 q = lds128(slot + u * kItemBytes + h * 512 + lane * 16);
          uint32_t bq[16];
          if (MODE == 0) {
            const uint32_t wv[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int k = 0; k < 4; ++k)
#pragma unroll
              for (int p = 0; p < 4; ++p) bq[4 * k + p] = ((wv[k] >> (4 * p)) & 0x000F000Fu) | 0x64006400u;
          } else {
            e2m1x8_to_f16x2x4(q.x, bq[0], bq[1], bq[2], bq[3]);
            e2m1x8_to_f16x2x4(q.y, bq[4], bq[5], bq[6], bq[7]);
            e2m1x8_to_f16x2x4(q.z, bq[8], bq[9], bq[10], bq[11]);
            e2m1x8_to_f16x2x4(q.w, bq[12], bq[13], bq[14], bq[15]);
          }
          // steps 0..3 (first 16 codes) and 4..7 as two independent accumulation chains
          float da[4], db[4];
          mma_f16_first(da, xa0.x, xa0.y, bq[0], bq[1]);
          mma_f16_first(db, xa2.x, xa2.y, bq[8], bq[9]);
          mma_f16(da, xa0.z, xa0.w, bq[2], bq[3]);
          mma_f16(db, xa2.z, xa2.w, bq[10], bq[11]);
          mma_f16(da, xa1.x, xa1.y, bq[4], bq[5]);
          mma_f16(db, xa3.x, xa3.y, bq[12], bq[13]);
          mma_f16(da, xa1.z, xa1.w, bq[6], bq[7]);
          mma_f16(db, xa3.z, xa3.w, bq[14], bq[15]);
          const uint32_t scv = sc[ss][u][h];
          if (MODE == 2) {
            const uint32_t sh = e4m3x2_to_f16x2(scv);
            const uint32_t s0 = __shfl_sync(0xffffffffu, sh, src0);
            const uint32_t s1 = __shfl_sync(0xffffffffu, sh, src1);
            acc[h][0] = fmaf(fmaf(da[0], f16_lo_to_f32(s0), db[0] * f16_hi_to_f32(s0)), xi, acc[h][0]);
            acc[h][1] = fmaf(fmaf(da[1], f16_lo_to_f32(s1), db[1] * f16_hi_to_f32(s1)), xi, acc[h][1]);
          } else if (MODE == 1) {
            const uint32_t s0 = __shfl_sync(0xffffffffu, scv, src0);
            const uint32_t s1 = __shfl_sync(0xffffffffu, scv, src1);
            acc[h][0] = fmaf(da[0] + db[0], e8m0_to_f32(s0) * xi, acc[h][0]);
            acc[h][1] = fmaf(da[1] + db[1], e8m0_to_f32(s1) * xi, acc[h][1]);
          } else {
            // D = sum (1024 + q) x  ->  s * (D - 1024 X) + b * X, X = sum of x over the chunk
            const uint32_t s0 = __shfl_sync(0xffffffffu, scv, src0);
            const uint32_t s1 = __shfl_sync(0xffffffffu, scv, src1);
            acc[h][0] = fmaf(fmaf(bf16_lo(s0), (da[0] + db[0]) - 1024.f * X, bf16_hi(s0) * X), xi, acc[h][0]);
            acc[h][1] = fmaf(fmaf(bf16_lo(s1), (da[1] + db[1]) - 1024.f * X, bf16_hi(s1) * X), xi, acc[h][1]);
          }
        }
      }
      if (++qs_c == SPR) { qs_c = 0; ++rg_c; }
    }
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  if (sb < se) flush();
  __syncthreads();
  const float unscale = (MODE == 2 && gs_w) ? __ldg(gs_w) : 1.0f;
  for (int r = tid; r < r1 - r0; r += kThreads) y[r0 + r] = (uint16_t)f32_to_bf16_rn(ypart[r] * unscale);
}

template <int MODE, bool QX>
cudaError_t launch_mode(const DevInfo& d, const uint16_t* x, const float* gs_x, const uint32_t* w,
                        const void* scales, const uint16_t* biases, const float* gs_w, int64_t N, int64_t K,
                        int group, uint16_t* y, cudaStream_t s) {
  const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(d.sm_count, (N + 7) / 8));
  const int64_t rows_max = (N + grid - 1) / grid;
  const int64_t rg_max = (rows_max + 15) / 16;
  const size_t smem = (size_t)kWarps * kRingBytes + (size_t)K * 2 + 64 + (size_t)(K / 32) * 8 +
                      (size_t)rg_max * 16 * 4;
  if (smem > d.smem_optin) return cudaErrorInvalidValue;
  {
    cudaError_t e = cudaFuncSetAttribute(qmv_kernel<MODE, QX>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, qmv_kernel<MODE, QX>, x, gs_x, w, scales, biases, gs_w, (int)N, (int)K, group, y);
}

}  // namespace

cudaError_t launch_qmv(const DevInfo& d, const uint16_t* x, const float* gs_x, int qx, const uint32_t* w,
                       const void* scales, const uint16_t* biases, const float* gs_w, int64_t N, int64_t K,
                       int mode, int group, uint16_t* y, int inject_timeout, cudaStream_t s) {
  // the tensor-core GEMV (NVFP4, MXFP4) needs K % 256 (NVFP4) or K % 512 (MXFP4) == 0,
  // 16-byte aligned scale rows and <= 256 rows per SM
  if ((mode == 2 || mode == 1) && (reinterpret_cast<uintptr_t>(scales) & 15) == 0 &&
      qmv_tc_supported(d, mode, N, K))
    return launch_qmv_tc(d, mode, x, gs_x, qx, w, static_cast<const uint8_t*>(scales), gs_w, N, K, y,
                         inject_timeout, s);
  if (mode == 0 && ((reinterpret_cast<uintptr_t>(scales) | reinterpret_cast<uintptr_t>(biases)) & 15) == 0 &&
      qmv_affine_supported(d, N, K, group))
    return launch_qmv_affine(d, x, w, static_cast<const uint16_t*>(scales), biases, N, K, group, y, s);
  if (mode == 2 && qx) return launch_mode<2, true>(d, x, gs_x, w, scales, biases, gs_w, N, K, group, y, s);
  if (mode == 1 && qx) return launch_mode<1, true>(d, x, gs_x, w, scales, biases, gs_w, N, K, group, y, s);
  if (mode == 2) return launch_mode<2, false>(d, x, nullptr, w, scales, biases, gs_w, N, K, group, y, s);
  if (mode == 1) return launch_mode<1, false>(d, x, nullptr, w, scales, biases, gs_w, N, K, group, y, s);
  return launch_mode<0, false>(d, x, nullptr, w, scales, biases, gs_w, N, K, group, y, s);
}

}  // namespace fp4
