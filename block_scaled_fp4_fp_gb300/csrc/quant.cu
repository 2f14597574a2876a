// quant.cu -- tensor amax / global scale, fp_quantize (NVFP4, MXFP4) and
// dequantize kernels.  All three stream HBM once and are bandwidth-bound.
//
// Pages: "perf(cuda): enable hardware NVFP4/MXFP4 conversion on Blackwell
// builds" (fp_quantize, the hardware e2m1x2 converter); "mlx 0.30.7.3 ->
// 0.30.7.6" qqmm.cpp quantize_input (packed uint32 codes, uint8 scales),
// qqmm_utils.h (128x4 scale tiles), quantized.cpp (fp_dequantize with the
// optional NVFP4 global scale).
#include <algorithm>

#include "common.cuh"
#include "launch.h"

namespace fp4 {

namespace {

constexpr int kThreads = 256;
constexpr int kQThreads = 64;
constexpr float kNvfp4MaxProduct = 2688.0f;  // 448 * 6

// ------------------------------------------------------------------ amax --
// Max of |x| over bf16 bit patterns: for non-NaN bf16 the order of
// (bits & 0x7FFF) as unsigned integers is the order of |x|, so the reduction is
// a packed 16-bit unsigned max on raw words.
__global__ void __launch_bounds__(kThreads) amax_partial_kernel(const uint16_t* __restrict__ x,
                                                                 int64_t n,
                                                                 uint32_t* __restrict__ partials) {
  asm volatile("griddepcontrol.wait;" ::: "memory");  // x may come from the previous kernel
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t nvec = n >> 3;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  uint32_t m2 = 0;
  const uint4* xv = reinterpret_cast<const uint4*>(x);
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + stride < nvec; i += 2 * stride) {
    uint4 a = ld_stream_v4(xv + i);
    uint4 b = ld_stream_v4(xv + i + stride);
    m2 = __vmaxu2(m2, a.x & 0x7FFF7FFFu);
    m2 = __vmaxu2(m2, a.y & 0x7FFF7FFFu);
    m2 = __vmaxu2(m2, a.z & 0x7FFF7FFFu);
    m2 = __vmaxu2(m2, a.w & 0x7FFF7FFFu);
    m2 = __vmaxu2(m2, b.x & 0x7FFF7FFFu);
    m2 = __vmaxu2(m2, b.y & 0x7FFF7FFFu);
    m2 = __vmaxu2(m2, b.z & 0x7FFF7FFFu);
    m2 = __vmaxu2(m2, b.w & 0x7FFF7FFFu);
  }
  for (; i < nvec; i += stride) {
    uint4 a = ld_stream_v4(xv + i);
    m2 = __vmaxu2(m2, a.x & 0x7FFF7FFFu);
    m2 = __vmaxu2(m2, a.y & 0x7FFF7FFFu);
    m2 = __vmaxu2(m2, a.z & 0x7FFF7FFFu);
    m2 = __vmaxu2(m2, a.w & 0x7FFF7FFFu);
  }
  uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
  if (blockIdx.x == 0 && threadIdx.x < (n & 7)) m = max(m, (uint32_t)(x[(nvec << 3) + threadIdx.x] & 0x7FFFu));
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ uint32_t red[kThreads / 32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kThreads / 32; ++w) m = max(m, red[w]);
    partials[blockIdx.x] = m;
  }
}

__global__ void __launch_bounds__(kThreads) amax_final_kernel(const uint32_t* __restrict__ partials,
                                                               int np, float* __restrict__ gs_out,
                                                               float* __restrict__ amax_out) {
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the partials of the kernel before
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  uint32_t m = 0;
  for (int i = threadIdx.x; i < np; i += blockDim.x) m = max(m, partials[i]);
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ uint32_t red[kThreads / 32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kThreads / 32; ++w) m = max(m, red[w]);
    const float amax = __uint_as_float(m << 16);
    *gs_out = __fdiv_rn(amax, kNvfp4MaxProduct);
    if (amax_out) *amax_out = amax;
  }
}

// -------------------------------------------------------------- quantize --
// One thread per block-scale group (16 or 32 bf16 = 2 or 4 16-byte loads), so
// the scale arithmetic (NVFP4: the division by a per-launch reciprocal and one
// correctly rounded reciprocal) runs once per group, for a batch of rows per
// thread (128 bytes of loads in flight).  Linear scales: blockIdx.x and
// threadIdx.x pick the group within a row, blockIdx.y strides over rows.
// 128x4-tiled scales: the mappings of quantize_nvfp4_tiled_kernel and
// quantize_tiled_kernel (below), which also write the tiles' zero padding.
// Codes leave as 8 or 16 contiguous bytes per thread.
// ------------------------------------------------- stochastic rounding --
// Random words: element e (row-major index) takes word e % 4 of Philox4x32-10
// (Salmon et al., "Parallel random numbers: as easy as 1, 2, 3") at the 128-bit
// counter offset + e / 4 under the key (seed low, seed high).
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t hi0 = __umulhi(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c;
}

__device__ __forceinline__ uint4 sr_words(uint64_t seed, uint64_t offset, uint64_t block) {
  const uint64_t b = offset + block;
  return philox4x32_10(make_uint4((uint32_t)b, (uint32_t)(b >> 32), b < offset ? 1u : 0u, 0u), (uint32_t)seed,
                       (uint32_t)(seed >> 32));
}

// Stochastic e2m1 rounding: |v| goes to one of its two grid neighbours lo < hi,
// up iff the top 24 bits of u are below floor(2^24 (|v| - lo) / (hi - lo));
// |v| >= 6 gives 6; the sign bit is kept.  Every step is exact in fp32.
__device__ __forceinline__ uint32_t e2m1_sr(float v, uint32_t u) {
  // branch-free (the three grid spacings are selected, not branched on, so a
  // warp's lanes never diverge): s = |v| / step is exact (step a power of 2),
  // lo = floor(s) step, frac = s - floor(s) = (|v| - lo) / step exactly
  const float a = fabsf(v);
  const bool r0 = a < 2.0f, r1 = a < 4.0f;
  const float inv = r0 ? 2.0f : (r1 ? 1.0f : 0.5f);
  const float s = __fmul_rn(a, inv);
  const float fl = floorf(s);
  const uint32_t f = __float2uint_rz(fl);
  const uint32_t li = r0 ? f : (r1 ? f + 2u : 6u);
  const float frac = __fsub_rn(s, fl);
  const uint32_t t = __float2uint_rz(__fmul_rn(frac, 16777216.0f));
  const uint32_t idx = (a < 6.0f) ? li + (((u >> 8) < t) ? 1u : 0u) : 7u;  // |v| >= 6 (or NaN): 6
  return idx | ((__float_as_uint(v) >> 28) & 8u);
}

template <int MODE, bool SR>
__device__ __forceinline__ void quantize_group(const uint4 (&v)[MODE == 2 ? 2 : 4], float gs, const Nvfp4Div& dv,
                                               uint32_t* __restrict__ xq_words,
                                               uint8_t* __restrict__ scale_byte, uint64_t e0,
                                               uint64_t seed, uint64_t offset) {
  constexpr int NV = (MODE == 2) ? 2 : 4;
  uint32_t m2 = 0;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    m2 = __vmaxu2(m2, v[i].x & 0x7FFF7FFFu);
    m2 = __vmaxu2(m2, v[i].y & 0x7FFF7FFFu);
    m2 = __vmaxu2(m2, v[i].z & 0x7FFF7FFFu);
    m2 = __vmaxu2(m2, v[i].w & 0x7FFF7FFFu);
  }
  const uint32_t mb = max(m2 & 0xFFFFu, m2 >> 16);
  float mul, sval;
  uint32_t sbyte;
  block_scale_rule<MODE>(mb, gs, dv, mul, sbyte, sval);
  uint32_t out[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const uint32_t wv[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
    uint32_t word = 0;
    if (SR) {  // 8 elements e0 + 8 i .. : two Philox blocks of four words
      const uint4 r0 = sr_words(seed, offset, (e0 >> 2) + 2 * i), r1 = sr_words(seed, offset, (e0 >> 2) + 2 * i + 1);
      const uint32_t u[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
#pragma unroll
      for (int j = 0; j < 4; ++j)
        word |= (e2m1_sr(__fmul_rn(bf16_lo(wv[j]), mul), u[2 * j]) |
                 (e2m1_sr(__fmul_rn(bf16_hi(wv[j]), mul), u[2 * j + 1]) << 4)) << (8 * j);
    } else {
      float f[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) fmul2_rn(bf16_lo(wv[j]), bf16_hi(wv[j]), mul, f[2 * j], f[2 * j + 1]);
      word = e2m1x8_rn(f);
    }
    out[i] = word;
  }
  if (MODE == 2) {
    *reinterpret_cast<uint2*>(xq_words) = make_uint2(out[0], out[1]);
  } else {
    *reinterpret_cast<uint4*>(xq_words) = make_uint4(out[0], out[1], out[2], out[3]);
  }
  *scale_byte = (uint8_t)sbyte;
}

// Linear scales: thread gi of the row quantizes group gi of RT rows (r, r + gy, ...).
template <int MODE, bool SR>
__global__ void __launch_bounds__(kQThreads) quantize_kernel(
    const uint16_t* __restrict__ x, int rows, int cols, const float* __restrict__ gs_ptr,
    uint32_t* __restrict__ xq, uint8_t* __restrict__ scales, uint64_t seed, uint64_t offset) {
  constexpr int G = (MODE == 2) ? 16 : 32;
  constexpr int NV = G / 8;
  constexpr int RT = (MODE == 2) ? 4 : 2;  // rows in flight per thread: 128 bytes of loads
  const int scols = cols / G;
  // programmatic dependent launch: this grid may start while the previous
  // kernel drains; x and the global scale are read only after it completed
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int gi = blockIdx.x * blockDim.x + threadIdx.x;  // group within the row
  if (gi >= scols) return;
  const float gs = (MODE == 2 && gs_ptr) ? __ldg(gs_ptr) : 1.0f;
  const Nvfp4Div dv = nvfp4_div(gs);  // the block-scale divisor's reciprocal, once per thread
  const int wpr = cols >> 3;  // code words per row
  const int gy = gridDim.y;
  for (int r = blockIdx.y; r < rows; r += RT * gy) {
    uint4 a[RT][NV];
#pragma unroll
    for (int k = 0; k < RT; ++k) {
      const int rk = r + k * gy;
      if (rk < rows) {
        const uint4* pa = reinterpret_cast<const uint4*>(x + (int64_t)rk * cols + gi * G);
#pragma unroll
        for (int i = 0; i < NV; ++i) a[k][i] = ld_stream_v4(pa + i);
      }
    }
#pragma unroll
    for (int k = 0; k < RT; ++k) {
      const int rk = r + k * gy;
      if (rk < rows)
        quantize_group<MODE, SR>(a[k], gs, dv, xq + (int64_t)rk * wpr + gi * NV, scales + (int64_t)rk * scols + gi,
                                 (uint64_t)rk * (uint64_t)cols + (uint64_t)gi * G, seed, offset);
    }
  }
}

// 128x4-tiled scales.  A block owns one tile column (groups 4 tc .. 4 tc + 3)
// of part of a 128-row tile: lane t of warp w in row batch b quantizes group
// 4 tc + t % 4 of row 128 tr + 32 q + rr, with q = (t / 4) % 4, rr = 2 slot +
// t / 16 and slot = part * 2 RT + w RT + b.  Within the tile that scale byte
// sits at rr * 16 + q * 4 + t % 4 = 32 slot + t, so one warp's 32 scale bytes
// of a batch are one 32-byte run, and each of its 8 rows reads 4 neighbouring
// groups of x.  The grid covers the padded buffer: rows past `rows` and groups
// past cols / G get zero bytes, so no other pass touches the padding.
template <int MODE, bool SR>
__global__ void __launch_bounds__(kQThreads) quantize_tiled_kernel(
    const uint16_t* __restrict__ x, int rows, int cols, const float* __restrict__ gs_ptr,
    uint32_t* __restrict__ xq, uint8_t* __restrict__ scales, int padded_cols, int ntr, uint64_t seed,
    uint64_t offset) {
  constexpr int G = (MODE == 2) ? 16 : 32;
  constexpr int NV = G / 8;
  constexpr int RT = (MODE == 2) ? 4 : 2;         // row batches in flight per thread: 128 bytes of loads
  constexpr int BPT = 32 / (4 * RT);              // blocks per 128-row tile (NVFP4 2, MXFP4 4)
  static_assert(kQThreads == 64, "two warps per block");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int scols = cols / G;
  const int t = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int c = (int)blockIdx.x * 4 + (t & 3);
  const int q = (t >> 2) & 3, hh = t >> 4;
  const int part = (int)(blockIdx.y % BPT);
  const float gs = (MODE == 2 && gs_ptr) ? __ldg(gs_ptr) : 1.0f;
  const Nvfp4Div dv = nvfp4_div(gs);
  const int wpr = cols >> 3;
  const int64_t tiles_per_row = padded_cols >> 2;
  for (int tr = (int)(blockIdx.y / BPT); tr < ntr; tr += (int)(gridDim.y / BPT)) {
    uint8_t* tile = scales + ((int64_t)tr * tiles_per_row + blockIdx.x) * 512;
    uint4 a[RT][NV];
#pragma unroll
    for (int b = 0; b < RT; ++b) {
      const int r = tr * 128 + 32 * q + 2 * (part * 2 * RT + w * RT + b) + hh;
      if (r < rows && c < scols) {
        const uint4* pa = reinterpret_cast<const uint4*>(x + (int64_t)r * cols + (int64_t)c * G);
#pragma unroll
        for (int i = 0; i < NV; ++i) a[b][i] = ld_stream_v4(pa + i);
      }
    }
#pragma unroll
    for (int b = 0; b < RT; ++b) {
      const int slot = part * 2 * RT + w * RT + b;
      const int r = tr * 128 + 32 * q + 2 * slot + hh;
      uint8_t* sb = tile + 32 * slot + t;
      if (r < rows && c < scols)
        quantize_group<MODE, SR>(a[b], gs, dv, xq + (int64_t)r * wpr + (int64_t)c * NV, sb,
                                 (uint64_t)r * (uint64_t)cols + (uint64_t)c * G, seed, offset);
      else
        *sb = 0;
    }
  }
}

// NVFP4 with 128x4-tiled scales.  Thread c of the row (a warp: 32 neighbouring
// groups, 1 KB of x per row) quantizes group c of the four rows 128 tr + rr +
// 32 q, q = 0..3, of one tile row: its four scale bytes are byte q*4 + c%4 of
// the 16-byte run rr*16 of tile (tr, c/4).  The four lanes of a tile column
// exchange them (a 4 x 4 byte transpose by shuffles) so that lane c writes the
// aligned word for q = c%4: one 4-byte store per lane instead of four bytes.
// The grid covers the padded buffer (zero bytes past `rows` and cols / 16).
template <bool SR>
__global__ void __launch_bounds__(kQThreads) quantize_nvfp4_tiled_kernel(
    const uint16_t* __restrict__ x, int rows, int cols, const float* __restrict__ gs_ptr,
    uint32_t* __restrict__ xq, uint8_t* __restrict__ scales, int padded_cols, int ntr, uint64_t seed,
    uint64_t offset) {
  constexpr int G = 16, NV = 2;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int scols = cols / G;
  const int c = (int)blockIdx.x * kQThreads + (int)threadIdx.x;
  const bool in_cols = c < scols, in_tiles = c < padded_cols;  // (uniform per 4-lane group)
  const int rr = (int)(blockIdx.y & 31u);
  const int lane = (int)(threadIdx.x & 31u), m = lane & 3;
  const float gs = gs_ptr ? __ldg(gs_ptr) : 1.0f;
  const Nvfp4Div dv = nvfp4_div(gs);
  const int wpr = cols >> 3;
  const int64_t tiles_per_row = padded_cols >> 2;
  const bool words_ok = (reinterpret_cast<uintptr_t>(scales) & 3u) == 0;
  for (int tr = (int)(blockIdx.y >> 5); tr < ntr; tr += (int)(gridDim.y >> 5)) {
    uint4 a[4][NV];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int r = tr * 128 + 32 * q + rr;
      if (r < rows && in_cols) {
        const uint4* pa = reinterpret_cast<const uint4*>(x + (int64_t)r * cols + (int64_t)c * G);
        a[q][0] = ld_stream_v4(pa);
        a[q][1] = ld_stream_v4(pa + 1);
      }
    }
    uint32_t packed = 0;  // byte q: this group's scale byte in row quadrant q
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int r = tr * 128 + 32 * q + rr;
      uint8_t sb = 0;
      if (r < rows && in_cols)
        quantize_group<2, SR>(a[q], gs, dv, xq + (int64_t)r * wpr + (int64_t)c * NV, &sb,
                              (uint64_t)r * (uint64_t)cols + (uint64_t)c * G, seed, offset);
      packed |= (uint32_t)sb << (8 * q);
    }
    // lane 4k + m collects byte m of its four neighbours' words (columns 4k .. 4k + 3)
    const int base = lane & ~3;
    const uint32_t v0 = __shfl_sync(0xffffffffu, packed, base);
    const uint32_t v1 = __shfl_sync(0xffffffffu, packed, base + 1);
    const uint32_t v2 = __shfl_sync(0xffffffffu, packed, base + 2);
    const uint32_t v3 = __shfl_sync(0xffffffffu, packed, base + 3);
    const uint32_t lo = __byte_perm(v0, v1, (uint32_t)(m | ((m + 4) << 4)));
    const uint32_t hi = __byte_perm(v2, v3, (uint32_t)(m | ((m + 4) << 4)));
    const uint32_t word = __byte_perm(lo, hi, 0x5410u);
    if (in_tiles) {
      uint8_t* dst = scales + ((int64_t)tr * tiles_per_row + (c >> 2)) * 512 + rr * 16 + m * 4;
      if (words_ok) {
        *reinterpret_cast<uint32_t*>(dst) = word;
      } else {  // a scale buffer that is not 4-byte aligned (uniform per launch)
#pragma unroll
        for (int k = 0; k < 4; ++k) dst[k] = (uint8_t)(word >> (8 * k));
      }
    }
  }
}

// ------------------------------------------------------------ dequantize --
// One thread per packed word (8 codes) -> one 16-byte store of 8 bf16.
template <int MODE>
__global__ void __launch_bounds__(kThreads) dequantize_kernel(
    const uint32_t* __restrict__ wq, const void* __restrict__ scales_v,
    const uint16_t* __restrict__ biases, int64_t rows, int64_t cols, int group,
    const float* __restrict__ gs_ptr, int tiled, int64_t padded_cols, uint16_t* __restrict__ out) {
  const int64_t nwords = rows * cols / 8;
  const int64_t wi = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (wi >= nwords) return;
  const uint32_t word = __ldg(wq + wi);
  const int64_t e0 = wi * 8;
  const int64_t r = e0 / cols, c = (e0 % cols) / group;
  const int64_t scols = cols / group;
  float v[8];
  if (MODE == 0) {
    const uint16_t* s16 = reinterpret_cast<const uint16_t*>(scales_v);
    const float s = __uint_as_float((uint32_t)__ldg(s16 + r * scols + c) << 16);
    const float b = __uint_as_float((uint32_t)__ldg(biases + r * scols + c) << 16);
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = __fadd_rn(__fmul_rn((float)((word >> (4 * j)) & 15u), s), b);
  } else {
    const uint8_t* s8 = reinterpret_cast<const uint8_t*>(scales_v);
    const int64_t off = tiled ? tiled_scale_offset(r, c, padded_cols) : r * scols + c;
    const uint32_t sb = __ldg(s8 + off);
    const float sc = (MODE == 2) ? e4m3_to_f32(sb) : e8m0_to_f32(sb);
    const float gs = (MODE == 2 && gs_ptr) ? __ldg(gs_ptr) : 1.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t h2 = e2m1x2_to_f16x2((word >> (8 * j)) & 0xFFu);
      const float lo = __fmul_rn(f16_lo_to_f32(h2), sc), hi = __fmul_rn(f16_hi_to_f32(h2), sc);
      v[2 * j] = (MODE == 2) ? __fmul_rn(lo, gs) : lo;
      v[2 * j + 1] = (MODE == 2) ? __fmul_rn(hi, gs) : hi;
    }
  }
  uint4 o;
  o.x = pack_bf16x2_rn(v[0], v[1]);
  o.y = pack_bf16x2_rn(v[2], v[3]);
  o.z = pack_bf16x2_rn(v[4], v[5]);
  o.w = pack_bf16x2_rn(v[6], v[7]);
  *reinterpret_cast<uint4*>(out + e0) = o;
}

}  // namespace

size_t amax_workspace_bytes(int64_t n) {
  (void)n;
  return 1024 * sizeof(uint32_t);
}

cudaError_t launch_amax(const DevInfo& d, const uint16_t* x, int64_t n, float* gs_out,
                        float* amax_out, uint32_t* partials, int max_partials, cudaStream_t s) {
  const int64_t nvec = (n + 7) / 8;
  int64_t blocks = (nvec + 2 * kThreads - 1) / (2 * kThreads);
  blocks = std::min<int64_t>(blocks, std::min<int64_t>(max_partials, (int64_t)d.sm_count * 4));
  blocks = std::max<int64_t>(blocks, 1);
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3((unsigned)blocks);
  cudaError_t e = cudaLaunchKernelEx(&cfg, amax_partial_kernel, x, n, partials);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3(1);
  return cudaLaunchKernelEx(&cfg, amax_final_kernel, (const uint32_t*)partials, (int)blocks, gs_out, amax_out);
}

cudaError_t launch_quantize(const DevInfo& d, const uint16_t* x, int64_t rows, int64_t cols,
                            int mode, int group, const float* gs, uint32_t* xq, uint8_t* scales,
                            int tiled, int sr, uint64_t seed, uint64_t offset, cudaStream_t s) {
  (void)d;
  const int64_t scols = cols / group;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kQThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int r = (int)rows, c = (int)cols;
  const float* g = (mode == 2) ? gs : nullptr;
  if (tiled) {
    // one block per (tile column, part of a 128-row tile); the loop strides over
    // tile rows only past 65535 blocks in y
    const int64_t pcol = ((scols + 3) / 4) * 4, ntr = (rows + 127) / 128;
    const int64_t bpt = (mode == 2) ? 2 : 4;
    const int64_t gy = std::max<int64_t>(1, std::min<int64_t>(ntr, 65535 / bpt)) * bpt;
    cfg.gridDim = dim3((unsigned)(pcol / 4), (unsigned)gy);
    const int pc = (int)pcol, nt = (int)ntr;
    if (mode == 2) {
      // one thread per group of a row, 32 rows (one per tile-row offset) per tile row in y
      const int64_t gy2 = std::max<int64_t>(1, std::min<int64_t>(ntr, 65535 / 32)) * 32;
      cfg.gridDim = dim3((unsigned)((pcol + kQThreads - 1) / kQThreads), (unsigned)gy2);
      return sr ? cudaLaunchKernelEx(&cfg, quantize_nvfp4_tiled_kernel<true>, x, r, c, g, xq, scales, pc, nt, seed,
                                     offset)
                : cudaLaunchKernelEx(&cfg, quantize_nvfp4_tiled_kernel<false>, x, r, c, g, xq, scales, pc, nt,
                                     (uint64_t)0, (uint64_t)0);
    }
    return sr ? cudaLaunchKernelEx(&cfg, quantize_tiled_kernel<1, true>, x, r, c, g, xq, scales, pc, nt, seed, offset)
              : cudaLaunchKernelEx(&cfg, quantize_tiled_kernel<1, false>, x, r, c, g, xq, scales, pc, nt,
                                   (uint64_t)0, (uint64_t)0);
  }
  // one batch of rows per thread (4 NVFP4 rows, 2 MXFP4 rows: 128 bytes of
  // loads in flight) and as many short-lived blocks as that takes -- measured
  // faster on this stream than fewer, longer-lived threads with software
  // pipelining; the loop strides over the rest only past 65535 row batches
  const int64_t rt = (mode == 2) ? 4 : 2;
  const int64_t gy = std::max<int64_t>(1, std::min<int64_t>((rows + rt - 1) / rt, 65535));
  cfg.gridDim = dim3((unsigned)((scols + kQThreads - 1) / kQThreads), (unsigned)gy);
  if (mode == 2)
    return sr ? cudaLaunchKernelEx(&cfg, quantize_kernel<2, true>, x, r, c, g, xq, scales, seed, offset)
              : cudaLaunchKernelEx(&cfg, quantize_kernel<2, false>, x, r, c, g, xq, scales, (uint64_t)0, (uint64_t)0);
  return sr ? cudaLaunchKernelEx(&cfg, quantize_kernel<1, true>, x, r, c, g, xq, scales, seed, offset)
            : cudaLaunchKernelEx(&cfg, quantize_kernel<1, false>, x, r, c, g, xq, scales, (uint64_t)0, (uint64_t)0);
}

cudaError_t launch_dequantize(const DevInfo& d, const uint32_t* wq, const void* scales,
                              const uint16_t* biases, int64_t rows, int64_t cols, int mode,
                              int group, const float* gs, int tiled, uint16_t* out,
                              cudaStream_t s) {
  (void)d;
  const int64_t nwords = rows * cols / 8;
  const unsigned grid = (unsigned)((nwords + kThreads - 1) / kThreads);
  const int64_t pcol = ((cols / group + 3) / 4) * 4;
  if (mode == 2)
    dequantize_kernel<2><<<grid, kThreads, 0, s>>>(wq, scales, biases, rows, cols, group, gs, tiled,
                                                   pcol, out);
  else if (mode == 1)
    dequantize_kernel<1><<<grid, kThreads, 0, s>>>(wq, scales, biases, rows, cols, group, gs, tiled,
                                                   pcol, out);
  else
    dequantize_kernel<0><<<grid, kThreads, 0, s>>>(wq, scales, biases, rows, cols, group, gs, 0,
                                                   pcol, out);
  return cudaGetLastError();
}

}  // namespace fp4
