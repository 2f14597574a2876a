// weight_stream.cu -- the NVFP4 GEMV's weight stream, with no GEMV.
//
// A measurement aid with no counterpart on the pages.  It moves NVFP4 weights
// (codes [N, K/2] bytes and linear E4M3 scales [N, K/16]) from HBM into shared
// memory the way the tensor-core qmv does -- one TMA box of R rows x 128 bytes
// of codes and one of R rows x 16 bytes of scales per K = 256 stage, a ring of
// slots holding what the GEMV's plan holds, the same split of K over the CTAs of a
// row block and the same rows per CTA, one CTA per SM, programmatic dependent
// launch with consumption after griddepcontrol.wait -- and computes nothing.
// Timed over the same weights, it is the launch-and-stream ceiling the GEMV
// is compared with: the part of a launch no kernel of this shape can avoid.
#include <algorithm>

#include "common.cuh"
#include "launch.h"

namespace fp4 {

namespace {

constexpr int kThreadsS = 64;                 // warp 0: TMA producer; warp 1: consumer
constexpr int kSlotsMax = 32;
constexpr uint32_t kSmemS = 226u * 1024u;   // + 512 bytes of static barriers <= 227 KB
constexpr uint32_t kRingS = kSmemS - 1024u;   // after aligning the base to 1024 bytes

__global__ void __launch_bounds__(kThreadsS, 1) weight_stream_kernel(const __grid_constant__ CUtensorMap tmW,
                                                                      const __grid_constant__ CUtensorMap tmS,
                                                                      int N, int K, int R, int split, int nslots,
                                                                      uint32_t wslot, uint32_t sslot,
                                                                      unsigned* __restrict__ err) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  __shared__ uint64_t full[kSlotsMax], empty[kSlotsMax];
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int rank = (int)(blockIdx.x % (unsigned)split);  // K slice of this CTA's row block
  const int blk = (int)(blockIdx.x / (unsigned)split), nblk = (int)(gridDim.x / (unsigned)split);
  const int r0 = (int)(((int64_t)N * blk) / nblk);
  const int kb0 = (int)(((int64_t)(K / 256) * rank) / split);
  const int nkb = (int)(((int64_t)(K / 256) * (rank + 1)) / split) - kb0;
  const uint32_t offS = (uint32_t)nslots * wslot;
  if (threadIdx.x < (unsigned)nslots) {
    mbar_init(&full[threadIdx.x], 1);
    mbar_init(&empty[threadIdx.x], 1);
  }
  fence_barrier_init();
  __syncthreads();
  bool failed = false;
  if (threadIdx.x == 0) {
    prefetch_tmap(&tmW);
    prefetch_tmap(&tmS);
    const uint32_t tx = (uint32_t)R * (128u + 16u);  // out-of-range rows are zero-filled and counted
    int s = 0, round = 0;
    for (int i = 0; i < nkb; ++i) {
      if (round > 0) mbar_wait(&empty[s], (round - 1) & 1, err, failed);
      mbar_arrive_expect_tx(&full[s], tx);
      tma_load_2d(smem + s * wslot, &tmW, &full[s], (kb0 + i) * 128, r0);
      tma_load_2d(smem + offS + s * sslot, &tmS, &full[s], (kb0 + i) * 16, r0);
      if (++s == nslots) { s = 0; ++round; }
    }
    // no copy may still be writing shared memory when the CTA exits (bounded
    // waits, even after an earlier one expired)
    bool drain_failed = false;
    for (int i = max(0, nkb - nslots); i < nkb; ++i)
      mbar_wait(&full[i % nslots], (i / nslots) & 1, err, drain_failed);
  } else if (threadIdx.x == 32) {
    asm volatile("griddepcontrol.wait;" ::: "memory");  // as the GEMV, which consumes after the previous kernel
    int s = 0, round = 0;
    for (int i = 0; i < nkb; ++i) {
      mbar_wait(&full[s], round & 1, err, failed);
      mbar_arrive(&empty[s]);
      if (++s == nslots) { s = 0; ++round; }
    }
  }
}

}  // namespace

cudaError_t launch_weight_stream(const DevInfo& d, const uint32_t* w, const uint8_t* scales, int64_t N,
                                 int64_t K, cudaStream_t s) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorInvalidValue;
  int split = 0, nblk = 0, R = 0, nslots = 0;
  if (!qmv_tc_geometry(d, N, K, &split, &nblk, &R, &nslots)) return cudaErrorInvalidValue;
  const int64_t grid = (int64_t)nblk * split;
  const uint32_t wslot = (uint32_t)((R + 7) / 8) * 1024u;
  const uint32_t sslot = ((uint32_t)R * 16u + 127u) / 128u * 128u;
  if ((uint32_t)nslots * (wslot + sslot) > kRingS || nslots > kSlotsMax) return cudaErrorInvalidValue;
  cuuint32_t estr[2] = {1, 1};
  CUtensorMap tmW, tmS;
  {
    cuuint64_t dims[2] = {(cuuint64_t)(K / 2), (cuuint64_t)N};
    cuuint64_t strides[1] = {(cuuint64_t)(K / 2)};
    cuuint32_t box[2] = {128, (cuuint32_t)R};
    if (fn(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint32_t*>(w), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    cuuint64_t dims[2] = {(cuuint64_t)(K / 16), (cuuint64_t)N};
    cuuint64_t strides[1] = {(cuuint64_t)(K / 16)};
    cuuint32_t box[2] = {16, (cuuint32_t)R};
    if (fn(&tmS, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(scales), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  cudaError_t e = cudaFuncSetAttribute(weight_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemS);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreadsS);
  cfg.dynamicSmemBytes = kSmemS;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, weight_stream_kernel, tmW, tmS, (int)N, (int)K, R, split, nslots, wslot, sslot,
                            d.err);
}

}  // namespace fp4
