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
constexpr float kNvfp4MaxProduct = 2688.0f;  // 448 * 6

// ------------------------------------------------------------------ amax --
// Max of |x| over bf16 bit patterns: for non-NaN bf16 the order of
// (bits & 0x7FFF) as unsigned integers is the order of |x|, so the reduction is
// a packed 16-bit unsigned max on raw words.
__global__ void __launch_bounds__(kThreads) amax_partial_kernel(const uint16_t* __restrict__ x,
                                                                 int64_t n,
                                                                 uint32_t* __restrict__ partials) {
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
// One thread per 16-byte chunk (8 bf16); a group is 2 (NVFP4) or 4 (MXFP4)
// neighbouring lanes, so the block amax is an in-thread max plus one or two
// xor-shuffles, and the codes leave as one coalesced uint32 per thread.
template <int MODE>
__global__ void __launch_bounds__(kThreads) quantize_kernel(
    const uint16_t* __restrict__ x, int64_t rows, int64_t cols, const float* __restrict__ gs_ptr,
    uint32_t* __restrict__ xq, uint8_t* __restrict__ scales, int tiled, int64_t padded_rows,
    int64_t padded_cols, int64_t main_blocks) {
  constexpr int G = (MODE == 2) ? 16 : 32;
  const int64_t scols = cols / G;
  if ((int64_t)blockIdx.x >= main_blocks) {
    // zero the padding bytes of the tiled scale buffer
    const int64_t total = padded_rows * padded_cols;
    for (int64_t off = ((int64_t)blockIdx.x - main_blocks) * blockDim.x + threadIdx.x; off < total;
         off += (int64_t)(gridDim.x - main_blocks) * blockDim.x) {
      const int64_t tile = off >> 9, within = off & 511;
      const int64_t r = (tile / (padded_cols >> 2)) * 128 + (within >> 4) + ((within & 15) >> 2) * 32;
      const int64_t c = (tile % (padded_cols >> 2)) * 4 + (within & 3);
      if (r >= rows || c >= scols) scales[off] = 0;
    }
    return;
  }
  const int64_t nchunks = rows * cols / 8;
  const int64_t ch = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const bool valid = ch < nchunks;
  uint4 v = make_uint4(0, 0, 0, 0);
  if (valid) v = ld_stream_v4(x + ch * 8);
  uint32_t mb = max(max(v.x & 0x7FFFu, (v.x >> 16) & 0x7FFFu), max(v.y & 0x7FFFu, (v.y >> 16) & 0x7FFFu));
  mb = max(mb, max(max(v.z & 0x7FFFu, (v.z >> 16) & 0x7FFFu), max(v.w & 0x7FFFu, (v.w >> 16) & 0x7FFFu)));
  mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
  if (MODE == 1) mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
  if (!valid) return;

  float f[8] = {bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y),
                bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w)};
  float mul;
  uint32_t sbyte;
  if (MODE == 2) {
    const float gs = gs_ptr ? __ldg(gs_ptr) : 1.0f;
    const float b = __uint_as_float(mb << 16);
    const float p = __fmul_rn(6.0f, gs);
    const float s = (b == 0.0f) ? 0.0f : __fdiv_rn(b, p);
    sbyte = e4m3_rn(s);
    const float d = __fmul_rn(e4m3_to_f32(sbyte), gs);
    mul = (d == 0.0f) ? 0.0f : __frcp_rn(d);
  } else {
    int se = -127;
    if (mb != 0) {
      const int E = (int)(mb >> 7);
      const int e = (E == 0) ? (-133 + (31 - __clz((int)(mb & 0x7Fu)))) : (E - 127);
      se = min(max(e - 2, -127), 127);
    }
    sbyte = (uint32_t)(se + 127);
    mul = exp2i_f32(-se);
  }
  uint32_t word = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    word |= e2m1x2_rn(__fmul_rn(f[2 * j], mul), __fmul_rn(f[2 * j + 1], mul)) << (8 * j);
  xq[ch] = word;
  if ((ch & (G / 8 - 1)) == 0) {
    const int64_t e0 = ch * 8;
    const int64_t r = e0 / cols, c = (e0 % cols) / G;
    const int64_t off = tiled ? tiled_scale_offset(r, c, padded_cols) : r * scols + c;
    scales[off] = (uint8_t)sbyte;
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
  amax_partial_kernel<<<(unsigned)blocks, kThreads, 0, s>>>(x, n, partials);
  amax_final_kernel<<<1, kThreads, 0, s>>>(partials, (int)blocks, gs_out, amax_out);
  return cudaGetLastError();
}

cudaError_t launch_quantize(const DevInfo& d, const uint16_t* x, int64_t rows, int64_t cols,
                            int mode, int group, const float* gs, uint32_t* xq, uint8_t* scales,
                            int tiled, cudaStream_t s) {
  (void)d;
  const int64_t nchunks = rows * cols / 8;
  const int64_t main_blocks = (nchunks + kThreads - 1) / kThreads;
  const int64_t scols = cols / group;
  const int64_t prow = ((rows + 127) / 128) * 128, pcol = ((scols + 3) / 4) * 4;
  int64_t pad_blocks = 0;
  if (tiled && (prow != rows || pcol != scols))
    pad_blocks = std::min<int64_t>((prow * pcol + kThreads - 1) / kThreads, 1024);
  const unsigned grid = (unsigned)(main_blocks + pad_blocks);
  if (mode == 2)
    quantize_kernel<2><<<grid, kThreads, 0, s>>>(x, rows, cols, gs, xq, scales, tiled, prow, pcol,
                                                 main_blocks);
  else
    quantize_kernel<1><<<grid, kThreads, 0, s>>>(x, rows, cols, nullptr, xq, scales, tiled, prow,
                                                 pcol, main_blocks);
  return cudaGetLastError();
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
