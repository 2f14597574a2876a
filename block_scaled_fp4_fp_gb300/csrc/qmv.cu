// qmv.cu -- M = 1 decode GEMV against 4-bit weights (affine, NVFP4, MXFP4).
//
// Pages: "epic: NVIDIA Volta (sm_70) inference acceleration program #1536"
// (Baseline: the decode step is the qmv weight stream; Diagnosis 3: the
// accumulator type -- here always fp32), "mlx 0.30.7.3 -> 0.30.7.6" qqmm.cpp
// (the M = 1 route through fp_qmv; W stored [N, K]).
//
// Layout of the work: x is staged once per CTA into shared memory as fp32
// (a 16-byte pad after every 32 values keeps the per-lane 128-byte strides
// free of bank conflicts); each warp owns one weight row at a time, its lanes
// stream the row as coalesced 16-byte vectors (32 codes = one chunk), several
// chunks in flight per lane, and the row sum is a warp-shuffle reduction.
// Per chunk the codes are decoded with the hardware e2m1x2 -> f16x2 converter,
// multiplied with x in fp32, and the block scale is applied once per group.
#include <algorithm>

#include "common.cuh"
#include "launch.h"

namespace fp4 {

namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kUnroll = 8;  // 16-byte chunks in flight per lane

__device__ __forceinline__ int xs_index(int k) { return k + ((k >> 5) << 2); }

// sum_{i<8} code_i * x_i over the 8 codes of `word`, x read from padded smem.
__device__ __forceinline__ float dot8(uint32_t word, const float* xp) {
  const float4 a = *reinterpret_cast<const float4*>(xp);
  const float4 b = *reinterpret_cast<const float4*>(xp + 4);
  const uint32_t h0 = e2m1x2_to_f16x2(word & 0xFFu);
  const uint32_t h1 = e2m1x2_to_f16x2((word >> 8) & 0xFFu);
  const uint32_t h2 = e2m1x2_to_f16x2((word >> 16) & 0xFFu);
  const uint32_t h3 = e2m1x2_to_f16x2(word >> 24);
  float s = f16_lo_to_f32(h0) * a.x;
  s = fmaf(f16_hi_to_f32(h0), a.y, s);
  s = fmaf(f16_lo_to_f32(h1), a.z, s);
  s = fmaf(f16_hi_to_f32(h1), a.w, s);
  s = fmaf(f16_lo_to_f32(h2), b.x, s);
  s = fmaf(f16_hi_to_f32(h2), b.y, s);
  s = fmaf(f16_lo_to_f32(h3), b.z, s);
  s = fmaf(f16_hi_to_f32(h3), b.w, s);
  return s;
}

// sum_{i<8} q_i * x_i for unsigned 4-bit q.
__device__ __forceinline__ float dot8_u4(uint32_t word, const float* xp) {
  const float4 a = *reinterpret_cast<const float4*>(xp);
  const float4 b = *reinterpret_cast<const float4*>(xp + 4);
  float s = (float)(word & 15u) * a.x;
  s = fmaf((float)((word >> 4) & 15u), a.y, s);
  s = fmaf((float)((word >> 8) & 15u), a.z, s);
  s = fmaf((float)((word >> 12) & 15u), a.w, s);
  s = fmaf((float)((word >> 16) & 15u), b.x, s);
  s = fmaf((float)((word >> 20) & 15u), b.y, s);
  s = fmaf((float)((word >> 24) & 15u), b.z, s);
  s = fmaf((float)(word >> 28), b.w, s);
  return s;
}

// MODE: 0 affine (group G in {32, 64, 128}), 1 MXFP4 (G = 32), 2 NVFP4 (G = 16).
template <int MODE>
__global__ void __launch_bounds__(kThreads) qmv_kernel(const uint16_t* __restrict__ x,
                                                        const uint32_t* __restrict__ w,
                                                        const void* __restrict__ scales_v,
                                                        const uint16_t* __restrict__ biases,
                                                        const float* __restrict__ gs_w, int N,
                                                        int K, int group,
                                                        uint16_t* __restrict__ y) {
  extern __shared__ float xs[];  // padded x (K + K/8 floats), then per-chunk sums of x (K/32)
  const int chunks = K >> 5;
  float* xsum = xs + K + (K >> 3);
  for (int v = threadIdx.x; v < (K >> 3); v += kThreads) {
    const uint4 q = __ldg(reinterpret_cast<const uint4*>(x) + v);
    const int k = v << 3;
    float4 a = make_float4(bf16_lo(q.x), bf16_hi(q.x), bf16_lo(q.y), bf16_hi(q.y));
    float4 b = make_float4(bf16_lo(q.z), bf16_hi(q.z), bf16_lo(q.w), bf16_hi(q.w));
    *reinterpret_cast<float4*>(xs + xs_index(k)) = a;
    *reinterpret_cast<float4*>(xs + xs_index(k) + 4) = b;
  }
  __syncthreads();
  if (MODE == 0) {
    for (int c = threadIdx.x; c < chunks; c += kThreads) {
      float s = 0.f;
      const float* p = xs + c * 36;
      for (int i = 0; i < 32; ++i) s += p[i];
      xsum[c] = s;
    }
    __syncthreads();
  }
  const int lane = threadIdx.x & 31;
  const int warp_global = blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int nwarps = gridDim.x * kWarps;
  const float gsw = (MODE == 2 && gs_w) ? __ldg(gs_w) : 1.0f;
  const int words = K >> 3;

  for (int n = warp_global; n < N; n += nwarps) {
    const uint32_t* wrow = w + (int64_t)n * words;
    float acc = 0.f;
    for (int c0 = lane; c0 < chunks; c0 += 32 * kUnroll) {
      uint4 q[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int c = c0 + 32 * u;
        q[u] = (c < chunks) ? ld_stream_v4(wrow + 4 * c) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int c = c0 + 32 * u;
        if (c >= chunks) break;
        const float* xp = xs + c * 36;
        if (MODE == 2) {
          const uint16_t sb = __ldg(reinterpret_cast<const uint16_t*>(
              reinterpret_cast<const uint8_t*>(scales_v) + (int64_t)n * (K >> 4) + 2 * c));
          const float s0 = e4m3_to_f32(sb & 0xFFu), s1 = e4m3_to_f32(sb >> 8);
          const float d0 = dot8(q[u].x, xp) + dot8(q[u].y, xp + 8);
          const float d1 = dot8(q[u].z, xp + 16) + dot8(q[u].w, xp + 24);
          acc = fmaf(d0, s0, acc);
          acc = fmaf(d1, s1, acc);
        } else if (MODE == 1) {
          const uint32_t sb = __ldg(reinterpret_cast<const uint8_t*>(scales_v) + (int64_t)n * (K >> 5) + c);
          const float d = (dot8(q[u].x, xp) + dot8(q[u].y, xp + 8)) +
                          (dot8(q[u].z, xp + 16) + dot8(q[u].w, xp + 24));
          acc = fmaf(d, e8m0_to_f32(sb), acc);
        } else {
          const int gi = (c << 5) / group;
          const int64_t si = (int64_t)n * (K / group) + gi;
          const float s = __uint_as_float((uint32_t)__ldg(reinterpret_cast<const uint16_t*>(scales_v) + si) << 16);
          const float b = __uint_as_float((uint32_t)__ldg(biases + si) << 16);
          const float d = (dot8_u4(q[u].x, xp) + dot8_u4(q[u].y, xp + 8)) +
                          (dot8_u4(q[u].z, xp + 16) + dot8_u4(q[u].w, xp + 24));
          acc = fmaf(d, s, acc);
          acc = fmaf(xsum[c], b, acc);
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) y[n] = (uint16_t)f32_to_bf16_rn(MODE == 2 ? acc * gsw : acc);
  }
}

template <int MODE>
cudaError_t launch_mode(const DevInfo& d, const uint16_t* x, const uint32_t* w, const void* scales,
                        const uint16_t* biases, const float* gs_w, int64_t N, int64_t K, int group,
                        uint16_t* y, cudaStream_t s) {
  const size_t smem = (size_t)(K + K / 8 + K / 32) * sizeof(float);
  if (smem > d.smem_optin) return cudaErrorInvalidValue;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(qmv_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
  }
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, qmv_kernel<MODE>, kThreads, smem);
  if (e != cudaSuccess) return e;
  per_sm = std::max(per_sm, 1);
  const int64_t want = (N + kWarps - 1) / kWarps;
  const int64_t grid = std::min<int64_t>(want, (int64_t)per_sm * d.sm_count);
  qmv_kernel<MODE><<<(unsigned)grid, kThreads, smem, s>>>(x, w, scales, biases, gs_w, (int)N, (int)K,
                                                          group, y);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_qmv(const DevInfo& d, const uint16_t* x, const uint32_t* w, const void* scales,
                       const uint16_t* biases, const float* gs_w, int64_t N, int64_t K, int mode,
                       int group, uint16_t* y, cudaStream_t s) {
  if (mode == 2) return launch_mode<2>(d, x, w, scales, biases, gs_w, N, K, group, y, s);
  if (mode == 1) return launch_mode<1>(d, x, w, scales, biases, gs_w, N, K, group, y, s);
  return launch_mode<0>(d, x, w, scales, biases, gs_w, N, K, group, y, s);
}

}  // namespace fp4
