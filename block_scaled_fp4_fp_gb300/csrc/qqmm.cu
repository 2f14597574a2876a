// qqmm.cu -- FP4 x FP4 block-scaled GEMM on the 5th-generation tensor cores.
//
// Pages: "mlx 0.30.7.3 -> 0.30.7.6" qqmm.cpp (QQMatmul::eval_gpu: x [M, K] and
// W [N, K] both K-major, W "always transposed", lda = ldb = K), qqmm_impl
// (block-scaled FP4 GEMM, batch 1, alpha/beta as device scalars),
// qqmm_utils.cu (alpha = amax_x*amax_w/(448*6)^2, beta = 0) and qqmm_utils.h
// (scales in 128-row x 4-column tiles, zero padded).
//
// Design (GB300-native, not the pages' cuBLASLt call).  Two persistent,
// warp-specialised kernels of 320 threads (warp 0 TMA producer, warp 1 tensor
// memory and MMA issue, warps 2-9 epilogue):
//   * qqmm_pair_kernel (every plain, batched and fused call): a cluster of two CTAs
//     on two SMs owns 256 x 256 output tiles and one thread issues
//     tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale (M 256, N 256, K 64;
//     4X with E4M3 scales for NVFP4, 2X with E8M0 for MXFP4), each CTA holding
//     its 128 x rows and half of the 256 W rows of every K = 256 stage, so an
//     SM moves 32 KB of codes per stage instead of 48 KB; a 5-stage ring; the
//     scale tiles go to tensor memory by tcgen05.cp (32x128b, replicated to
//     the four lane quadrants -- the 128x4 tile is exactly that copy's source
//     layout); the epilogue drains the fp32 accumulator (tcgen05.ld), scales
//     by alpha, rounds to bf16, releases the accumulator to the next tile's
//     MMAs and writes through a swizzled shared-memory stage with TMA tensor
//     stores.
//   * the fused quantized-activation call (qqmm_quantize_x) launches the pair
//     kernel cooperatively with clusters of two: a quantize prologue (below)
//     writes x's codes and tiled scales before the mainloop reads them;
//   * qqmm_kernel (the fallback when no CTA pair can be resident): one CTA per
//     SM, 128 x 256 tiles, tcgen05 cta_group::1, a 4-stage ring, scale tiles
//     by 1-D bulk copies, per-thread row stores.
//   * every mbarrier wait is bounded; an expired wait records an error word
//     and the protocol continues, so the kernels always terminate.
#include <algorithm>
#include <mutex>
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "launch.h"
#include "pair.cuh"

namespace fp4 {

namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 256;             // fp4 elements per stage (128 bytes per row)
constexpr int BK_BYTES = BK / 2;
constexpr int STAGES = 4;
constexpr int kEpiWarps = 8;
constexpr int kThreads = (2 + kEpiWarps) * 32;  // producer, MMA, 8 epilogue warps
constexpr uint32_t A_BYTES = BM * BK_BYTES;  // 16 KB
constexpr uint32_t B_BYTES = BN * BK_BYTES;  // 32 KB
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COL = 0;     // accumulator: columns [0, 256)
constexpr uint32_t SF_COL = 256;    // scale factors: 48 columns per stage

template <int MODE>
struct Cfg {
  static constexpr int GROUP = (MODE == 2) ? 16 : 32;
  // 128x4 scale tiles per 128 rows per stage (K = 256 covers 256/GROUP scale columns)
  static constexpr int TILES_PER_STAGE = (BK / GROUP) / 4;         // 4 (NVFP4) or 2 (MXFP4)
  static constexpr uint32_t SFA_BYTES = TILES_PER_STAGE * 512;     // one 128-row tile
  static constexpr uint32_t SFB_BYTES = 2 * SFA_BYTES;             // two 128-row tiles
  static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
  static constexpr uint32_t SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/;
  // instruction descriptor: a/b format E2M1 (1), K-major, N>>3, M>>4, scale format
  static constexpr uint32_t IDESC = (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                                    ((MODE == 2 ? 0u : 1u) << 23) | ((uint32_t)(BM >> 4) << 24);
};

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row atoms of
// 1024 bytes (stride byte offset), descriptor version 1.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Descriptor of one 512-byte scale tile: 32 rows x 16 bytes, no swizzle,
// 8-row core matrices 128 bytes apart.
__device__ __forceinline__ uint64_t desc_sf(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(128 >> 4) << 32) | ((uint64_t)1 << 46);
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               :: "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void tc_cp_sf(uint32_t tmem, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" :: "r"(tmem), "l"(sdesc) : "memory");
}

template <int MODE>
__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                       uint32_t sfb, uint32_t accumulate) {
  if (MODE == 2) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
        :: "r"(d), "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate) : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
        :: "r"(d), "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate) : "memory");
  }
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

// 32 lanes x 64 consecutive 32-bit columns (one register per column)
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, "
      "%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, "
      "%48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
        "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
        "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Batch b of a batched call reads its x codes at z = b (x) and z = b * wz (W:
// wz = 0 when every batch shares W), its scale tiles at b * stride_sx and
// b * stride_sw bytes, its global scales gs_x[b], gs_w[b], and writes out + b *
// stride_out.
struct Batch {
  int count = 1;
  int wz = 1;
  int64_t stride_sx = 0, stride_sw = 0, stride_out = 0;
};

// The quantized-activation prologue of a fused call: bf16 x [M, K] is
// quantized by every CTA of the (co-resident, cooperative) grid into the
// caller's workspace -- codes xq and the 128x4-tiled scales sx the GEMM then
// reads -- after, when no activation global scale is given (NVFP4), the tensor
// amax reduced across the grid.  Grid barriers use one word, bar[0] (arrival
// count and generation bit; zero before the first call, and each barrier
// leaves the count at zero); their waits are bounded.
struct FusedX {
  const uint16_t* x = nullptr;
  const float* gs_in = nullptr;  // NVFP4 activation global scale, or nullptr: amax / 2688 from x
  float* gs_out = nullptr;       // the global scale used, for the epilogue (workspace)
  float* gs_user = nullptr;      // and a copy for the caller (nullable)
  uint32_t* xq = nullptr;
  uint8_t* sx = nullptr;
  uint32_t* partials = nullptr;  // one per CTA
  unsigned* bar = nullptr;
  int padded_rows = 0, padded_cols = 0;
};

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned atom_add_acq_rel_gpu(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ void red_add_release_gpu(unsigned* p, unsigned v) {
  asm volatile("red.add.release.gpu.global.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

// All CTAs of the grid meet on one word, bar[0]: the arrival count in bits 0-30
// and a generation in bit 31.  Thread 0 of each CTA arrives with one
// acquire-release add (its CTA's writes, ordered before it by the CTA barrier,
// are released; the last arrival acquires everyone's).  The last arrival clears
// the count and flips the generation with a single release add (count n -> 0
// and bit 31 toggled, modulo 2^32); the others wait (bounded) for the flip.  A
// zero-filled word is a valid start and every barrier leaves the count at 0.
__device__ void grid_barrier(unsigned* bar, unsigned* err, bool& failed) {
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned n = gridDim.x;
    const unsigned old = atom_add_acq_rel_gpu(bar, 1u);
    const unsigned gen = old & 0x80000000u;
    if ((old & 0x7fffffffu) == n - 1) {
      red_add_release_gpu(bar, 0x80000000u - n);
    } else if (!failed) {
      const long long t0 = clock64();
      while ((ld_acquire_gpu(bar) & 0x80000000u) == gen) {
        if (clock64() - t0 > kWaitLimitCycles) {
          record_error(err, kErrTimeout);
          failed = true;
          break;
        }
      }
    }
  }
  __syncthreads();
}

// 16 bytes from shared memory (32-bit shared address)
__device__ __forceinline__ uint4 lds_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

// The fused activation quantize that runs before the GEMM in a cooperative
// launch (all CTAs resident).  CTA b owns a contiguous share of x's scale
// groups and moves it through the idle operand ring (`ring`, `ring_bytes`) in
// NB chunks by bulk copies, so that a whole ring of bytes is in flight per SM:
//   1. NVFP4 without a given activation scale: max |x| of the share from
//      shared memory, one partial per CTA, a grid barrier, gs = amax / 2688
//      ("NVFP4 and MXFP4 formats", the tensor-level scale);
//   2. quantize every group of the share (the block-scale rule of the format,
//      e2m1 rounding to nearest even) into codes and 128x4-tiled scales.
// The chunks still in the ring after step 1 (all of them when the share fits)
// are quantized first and are not read again from global memory.
template <int MODE>
__device__ void quantize_prologue(const FusedX& fx, int M, int K, uint8_t* ring, uint32_t ring_bytes,
                                  unsigned* err, bool& failed) {
  constexpr int G = (MODE == 2) ? 16 : 32;
  constexpr int GB = 2 * G;  // bytes of x per scale group
  constexpr int NV = G / 8;  // 16-byte pieces per group
  constexpr int NB = 4;      // chunk buffers
  __shared__ uint32_t red[kThreads / 32];
  __shared__ float gs_sh;
  __shared__ uint64_t cbar[NB];
  const int T = (int)blockDim.x;
  const int scols = K / G;
  const int64_t ngroups = (int64_t)M * scols;
  const int64_t g_lo = ngroups * blockIdx.x / gridDim.x;
  const int64_t share = ngroups * (blockIdx.x + 1) / gridDim.x - g_lo;
  const int gpc = (int)(ring_bytes / NB / GB);  // groups per chunk
  const uint32_t CH = (uint32_t)gpc * GB;
  const int nchunks = (int)((share + gpc - 1) / gpc);
  const uint8_t* xs = reinterpret_cast<const uint8_t*>(fx.x) + g_lo * GB;
  const uint32_t ring_s = smem_u32(ring);
  auto chunk_groups = [&](int j) { return (int)min((int64_t)gpc, share - (int64_t)j * gpc); };
  auto issue = [&](int j, int b) {  // one thread: chunk j of the share into buffer b
    const uint32_t bytes = (uint32_t)chunk_groups(j) * GB;
    mbar_arrive_expect_tx(&cbar[b], bytes);
    bulk_load(ring + (size_t)b * CH, xs + (int64_t)j * gpc * GB, bytes, &cbar[b]);
  };
  if (threadIdx.x == 0) {
    for (int b = 0; b < NB; ++b) mbar_init(&cbar[b], 1);
    fence_barrier_init();
  }
  __syncthreads();
  uint32_t phase = 0;  // bit b: parity of buffer b's next completion
  float gs = 1.0f;
  int nres = 0;        // chunks left in the ring by the max pass
  if (MODE == 2 && fx.gs_in) {
    gs = __ldg(fx.gs_in);
  } else if (MODE == 2) {
    // tensor amax over bf16 magnitude bits (their unsigned order is |x|'s order)
    if (threadIdx.x == 0)
      for (int j = 0; j < min(NB, nchunks); ++j) issue(j, j);
    uint32_t m = 0;
    for (int j = 0; j < nchunks; ++j) {
      const int b = j % NB;
      mbar_wait(&cbar[b], (phase >> b) & 1u, err, failed);
      phase ^= 1u << b;
      const uint32_t src = ring_s + (uint32_t)b * CH;
      const int nv = chunk_groups(j) * NV;
      int i = threadIdx.x;
      for (; i + 3 * T < nv; i += 4 * T) {  // four independent loads per round
        uint4 a[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) a[u] = lds_v4(src + 16u * (uint32_t)(i + u * T));
#pragma unroll
        for (int u = 0; u < 4; ++u) m = max(m, max_mag8(a[u]));
      }
      for (; i < nv; i += T) m = max(m, max_mag8(lds_v4(src + 16u * (uint32_t)i)));
      if (j + NB < nchunks) {
        __syncthreads();  // buffer b read by every thread
        if (threadIdx.x == 0) issue(j + NB, b);
      }
    }
    nres = min(NB, nchunks);
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int w = 1; w < kThreads / 32; ++w) m = max(m, red[w]);
      fx.partials[blockIdx.x] = m;
    }
    grid_barrier(fx.bar, err, failed);
    // every thread reads its share of the per-CTA maxima (one L2 round trip, not gridDim.x)
    uint32_t a = 0;
    for (unsigned b = threadIdx.x; b < gridDim.x; b += blockDim.x) a = max(a, __ldcg(fx.partials + b));
    for (int o = 16; o > 0; o >>= 1) a = max(a, __shfl_xor_sync(0xffffffffu, a, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = a;
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int w = 1; w < kThreads / 32; ++w) a = max(a, red[w]);
      gs_sh = __fdiv_rn(__uint_as_float(a << 16), 2688.0f);
      if (blockIdx.x == 0) {
        *fx.gs_out = gs_sh;
        if (fx.gs_user) *fx.gs_user = gs_sh;
      }
    }
    __syncthreads();
    gs = gs_sh;
  }
  if (MODE == 2 && fx.gs_in && blockIdx.x == 0 && threadIdx.x == 0) {
    *fx.gs_out = gs;
    if (fx.gs_user) *fx.gs_user = gs;
  }
  // quantize: one thread per group.  A thread reads its group's 16-byte pieces
  // in an order rotated by its lane so that eight neighbouring threads' reads
  // fall in distinct shared-memory banks.
  constexpr int U = (MODE == 2) ? 4 : 2;
  const Nvfp4Div dv = nvfp4_div(gs);  // the block-scale divisor's reciprocal, once per thread
  const int dr = T / scols, dc = T % scols;
  const uint32_t rot = (MODE == 2) ? ((threadIdx.x >> 2) & 1u) : ((threadIdx.x >> 1) & 3u);
  const int base = nres > 0 ? (nchunks - nres) % NB : 0;
  if (threadIdx.x == 0 && nres == 0)
    for (int p = 0; p < min(NB, nchunks); ++p) issue(p, p);
  for (int p = 0; p < nchunks; ++p) {
    // the chunks left by the max pass come first, then the share from its start
    const int b = (base + p) % NB;
    const int j = p < nres ? nchunks - nres + p : p - nres;
    if (p >= nres) {
      mbar_wait(&cbar[b], (phase >> b) & 1u, err, failed);
      phase ^= 1u << b;
    }
    const int cnt = chunk_groups(j);
    const int64_t g0 = g_lo + (int64_t)j * gpc + threadIdx.x;
    int r = (int)(g0 / scols), c = (int)(g0 % scols);
    const uint32_t src = ring_s + (uint32_t)b * CH;
    for (int l0 = threadIdx.x; l0 < cnt; l0 += U * T) {
      // U independent groups per round (l0 + u T), for instruction-level parallelism
      uint4 v[U][NV];
      int rr[U], cc[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        rr[u] = r;
        cc[u] = c;
        c += dc;
        r += dr;
        if (c >= scols) {
          c -= scols;
          ++r;
        }
        if (l0 + u * T < cnt) {
#pragma unroll
          for (int k = 0; k < NV; ++k)
            v[u][k] = lds_v4(src + (uint32_t)(l0 + u * T) * GB + 16u * ((k + rot) & (NV - 1)));
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (l0 + u * T >= cnt) continue;
        uint32_t mb = 0;
#pragma unroll
        for (int k = 0; k < NV; ++k) mb = max(mb, max_mag8(v[u][k]));
        float mul, sval;
        uint32_t sbyte;
        block_scale_rule<MODE>(mb, gs, dv, mul, sbyte, sval);
        uint32_t w[NV];
#pragma unroll
        for (int k = 0; k < NV; ++k) {
          const uint32_t wv[4] = {v[u][k].x, v[u][k].y, v[u][k].z, v[u][k].w};
          float f[8];
#pragma unroll
          for (int q = 0; q < 4; ++q) fmul2_rn(bf16_lo(wv[q]), bf16_hi(wv[q]), mul, f[2 * q], f[2 * q + 1]);
          w[k] = e2m1x8_rn(f);
        }
        // piece i's codes are w[(i - rot) mod NV]
        uint32_t* dst = fx.xq + (int64_t)rr[u] * (K / 8) + (int64_t)cc[u] * NV;
        if constexpr (NV == 2) {
          *reinterpret_cast<uint2*>(dst) = rot ? make_uint2(w[1], w[0]) : make_uint2(w[0], w[1]);
        } else {
          uint32_t a[4], o[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) a[i] = (rot & 1u) ? w[(i + 3) & 3] : w[i];
#pragma unroll
          for (int i = 0; i < 4; ++i) o[i] = (rot & 2u) ? a[(i + 2) & 3] : a[i];
          *reinterpret_cast<uint4*>(dst) = make_uint4(o[0], o[1], o[2], o[3]);
        }
        fx.sx[tiled_scale_offset(rr[u], cc[u], fx.padded_cols)] = (uint8_t)sbyte;
      }
    }
    if (p + NB < nchunks) {
      __syncthreads();  // buffer b read by every thread
      if (threadIdx.x == 0) issue(p + NB - nres, b);
    }
  }
  // the padding rows of the scale tiles are zero
  const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t pad = (int64_t)(fx.padded_rows - M) * fx.padded_cols;
  for (int64_t i = tid; i < pad; i += nthreads) {
    const int r = M + (int)(i / fx.padded_cols), c = (int)(i % fx.padded_cols);
    fx.sx[tiled_scale_offset(r, c, fx.padded_cols)] = 0;
  }
  // generic-proxy writes, read next by TMA and bulk copies (async proxy) in
  // other CTAs; the ring, read here, is written next by the GEMM's TMA loads
  asm volatile("fence.proxy.async.global;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  grid_barrier(fx.bar, err, failed);
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

template <int MODE, bool FQ>
__global__ void __launch_bounds__(kThreads, 1) qqmm_kernel(
    const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
    const uint8_t* __restrict__ sx, const uint8_t* __restrict__ sw, const float* __restrict__ gs_x,
    const float* __restrict__ gs_w, int M, int N, int K, Batch bt, uint16_t* __restrict__ out,
    unsigned* __restrict__ err, int inject_timeout, FusedX fx) {
  using C = Cfg<MODE>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  // per stage: [A | B | SFA | SFB]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * C::STAGE_BYTES);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* acc_full = bars + 2 * STAGES;
  uint64_t* acc_empty = bars + 2 * STAGES + 1;
  uint64_t* never = bars + 2 * STAGES + 2;  // fault-injection barrier, never arrived at
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 3);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_kb = K / BK;
  const int num_m = (M + BM - 1) / BM, num_n = (N + BN - 1) / BN;
  const int tiles_per_batch = num_m * num_n;
  const int num_tiles = tiles_per_batch * bt.count;
  const int64_t tiles_per_rowtile = (K / C::GROUP) / 4;  // 128x4 scale tiles along K
  const int n_rowtiles = (N + 127) / 128;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, kEpiWarps);
    mbar_init(never, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(tmem_slot)), "r"(TMEM_COLS) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool failed = false;  // this thread gave up a wait (see mbar_wait)
  if (FQ) quantize_prologue<MODE>(fx, M, K, smem, STAGES * C::STAGE_BYTES, err, failed);

  if (warp == 0) {
    // ------------------------------------------------------------ producer --
    if (elect_one_sync()) {
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmB);
      int g = 0;  // k-blocks issued by this CTA so far (ring position)
      for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
        const int b = tile / tiles_per_batch, rem = tile - b * tiles_per_batch;
        const int m_blk = rem % num_m, n_blk = rem / num_m;
        const uint8_t* sxb = sx + (int64_t)b * bt.stride_sx;
        const uint8_t* swb = sw + (int64_t)b * bt.stride_sw;
        const bool second_b_tile = (n_blk * 2 + 1) < n_rowtiles;
        const uint32_t tx = A_BYTES + B_BYTES + C::SFA_BYTES + (second_b_tile ? 2u : 1u) * C::SFA_BYTES;
        for (int kb = 0; kb < num_kb; ++kb, ++g) {
          const int s = g % STAGES;
          const int round = g / STAGES;
          if (round > 0) mbar_wait(&empty[s], (round - 1) & 1, err, failed);
          uint8_t* st = smem + s * C::STAGE_BYTES;
          mbar_arrive_expect_tx(&full[s], tx);
          tma_load_3d(st, &tmA, &full[s], kb * BK_BYTES, m_blk * BM, b);
          tma_load_3d(st + A_BYTES, &tmB, &full[s], kb * BK_BYTES, n_blk * BN, b * bt.wz);
          const int64_t tcol = (int64_t)kb * C::TILES_PER_STAGE;
          bulk_load(st + A_BYTES + B_BYTES, sxb + ((int64_t)m_blk * tiles_per_rowtile + tcol) * 512,
                    C::SFA_BYTES, &full[s]);
          bulk_load(st + A_BYTES + B_BYTES + C::SFA_BYTES,
                    swb + ((int64_t)(2 * n_blk) * tiles_per_rowtile + tcol) * 512, C::SFA_BYTES, &full[s]);
          if (second_b_tile)
            bulk_load(st + A_BYTES + B_BYTES + 2 * C::SFA_BYTES,
                      swb + ((int64_t)(2 * n_blk + 1) * tiles_per_rowtile + tcol) * 512, C::SFA_BYTES,
                      &full[s]);
        }
      }
      // drain: every stage's last fill has landed before the CTA may exit (the
      // waits run, bounded, even after an earlier one expired)
      bool drain_failed = false;
      for (int k = (g > STAGES ? g - STAGES : 0); k < g; ++k)
        mbar_wait(&full[k % STAGES], (k / STAGES) & 1, err, drain_failed);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer --
    if (elect_one_sync()) {
      if (inject_timeout) {
        bool injected = false;  // separate flag: the injected expiry must not stop later waits
        mbar_wait(never, 0, err, injected, 2000000LL);
      }
      int g = 0, it = 0;
      for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++it) {
        // the epilogue must have read the previous tile's accumulator
        if (it > 0) mbar_wait(acc_empty, (it - 1) & 1, err, failed);
        tc_fence_after();
        for (int kb = 0; kb < num_kb; ++kb, ++g) {
          const int s = g % STAGES;
          mbar_wait(&full[s], (g / STAGES) & 1, err, failed);
          tc_fence_after();
          const uint32_t st = base + s * C::STAGE_BYTES;
          const uint32_t sfa_smem = st + A_BYTES + B_BYTES;
          const uint32_t sfb_smem = sfa_smem + C::SFA_BYTES;
          const uint32_t sfa_t = tmem + SF_COL + s * 48;
          const uint32_t sfb_t = sfa_t + 16;
#pragma unroll
          for (int j = 0; j < C::TILES_PER_STAGE; ++j) {
            tc_cp_sf(sfa_t + 4 * j, desc_sf(sfa_smem + 512 * j));
            tc_cp_sf(sfb_t + 8 * j, desc_sf(sfb_smem + 512 * j));
            tc_cp_sf(sfb_t + 8 * j + 4, desc_sf(sfb_smem + C::SFA_BYTES + 512 * j));
          }
          const uint64_t adesc = desc_sw128(st);
          const uint64_t bdesc = desc_sw128(st + A_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 64; ++k) {
            // K = 64 fp4 = 32 bytes further along the swizzled 128-byte row
            const int tl = (MODE == 2) ? k : (k >> 1);
            const uint32_t sf_id = (MODE == 2) ? 0u : (uint32_t)((k & 1) * 2);
            const uint32_t idesc = C::IDESC | (sf_id << 29) | (sf_id << 4);
            tc_mma<MODE>(tmem + ACC_COL, adesc + (uint64_t)(2 * k), bdesc + (uint64_t)(2 * k), idesc,
                         sfa_t + 4 * tl, sfb_t + 8 * tl, (kb > 0 || k > 0) ? 1u : 0u);
          }
          tc_commit(&empty[s]);
        }
        tc_commit(acc_full);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue --
    // 8 warps: lane quadrant q = warp % 4 (tensor-memory access rule), column half h.
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;
    int it = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++it) {
      const int b = tile / tiles_per_batch, rem = tile - b * tiles_per_batch;
      const int m_blk = rem % num_m, n_blk = rem / num_m;
      // (a fused call's activation scale was written by this grid: read it coherently)
      const float gx = gs_x ? (FQ ? __ldcg(gs_x + b) : __ldg(gs_x + b)) : 1.0f;
      const float alpha = __fmul_rn(gx, gs_w ? __ldg(gs_w + b) : 1.0f);
      mbar_wait(acc_full, it & 1, err, failed);
      tc_fence_after();
      // drain this warp's 32 rows x 128 columns into registers as packed bf16
      uint32_t o[64];
#pragma unroll
      for (int c4 = 0; c4 < 2; ++c4) {
        uint32_t r[4][16];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + ACC_COL + h * 128 + (c4 * 4 + j) * 16, r[j]);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
          for (int e = 0; e < 8; ++e)
            o[(c4 * 4 + j) * 8 + e] = pack_bf16x2_rn(__fmul_rn(__uint_as_float(r[j][2 * e]), alpha),
                                                     __fmul_rn(__uint_as_float(r[j][2 * e + 1]), alpha));
      }
      // the accumulator may now be overwritten by the next tile's MMAs
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty);
      const int row = m_blk * BM + 32 * q + lane;
      if (row < M) {
        uint16_t* orow = out + (int64_t)b * bt.stride_out + (int64_t)row * N + n_blk * BN + h * 128;
        const int cols_left = N - (n_blk * BN + h * 128);
#pragma unroll
        for (int v = 0; v < 16; ++v)
          if (8 * v < cols_left)
            *reinterpret_cast<uint4*>(orow + 8 * v) = make_uint4(o[4 * v], o[4 * v + 1], o[4 * v + 2], o[4 * v + 3]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(TMEM_COLS) : "memory");
  }
}

// ---------------------------------------------------------------------------
// CTA-pair variant (tcgen05 cta_group::2).  A cluster of two CTAs on two SMs
// owns a 256 x 256 output tile: CTA r holds rows [128 r, 128 r + 128) of the
// x tile and rows [128 r, 128 r + 128) of the W tile in its shared memory, and
// one thread of CTA 0 issues M = 256 MMAs that read both CTAs' operands and
// accumulate each CTA's 128 rows x 256 columns in that CTA's tensor memory.
// Each SM so loads and reads 32 KB of codes per K = 256 stage instead of 48 KB
// for the same 128 x 256 x 256 products.
//   * both CTAs' loads complete on CTA 0's `full` barrier (TMA .cta_group::2,
//     the barrier addressed in CTA 0 through mapa); CTA 0's producer expects
//     both CTAs' bytes;
//   * CTA 0's MMA thread releases a stage in both CTAs (commit multicast to
//     their `empty` barriers) and publishes the accumulator to both epilogues;
//   * the epilogue warps of both CTAs arrive on CTA 0's `acc_empty`;
//   * scale tiles arrive by TMA too (a 4-D view of the 128x4-tiled bytes) so
//     that they can complete on CTA 0's barrier; tcgen05.cp.cta_group::2
//     moves each CTA's scale tiles into its own tensor memory.  Each CTA
//     holds the scales of its own x rows and of all 256 W rows.
constexpr int kPairStages = 5;

template <int MODE>
struct PairCfg {
  static constexpr int TPS = Cfg<MODE>::TILES_PER_STAGE;
  static constexpr uint32_t SF_BYTES = TPS * 512;       // one 128-row scale tile slice
  static constexpr uint32_t AB_BYTES = 2 * A_BYTES;      // x rows + half the W rows: 32 KB
  static constexpr uint32_t STAGE_BYTES = AB_BYTES + 3 * SF_BYTES;  // + SFA + two SFB slices
  static constexpr uint32_t TX_CTA = STAGE_BYTES;        // bytes one CTA loads per stage
  static constexpr uint32_t SMEM_BYTES = kPairStages * STAGE_BYTES + kEpiWarps * 4096 + 1024 + 256;
  static constexpr uint32_t IDESC = (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                                    ((MODE == 2 ? 0u : 1u) << 23) | ((uint32_t)(256 >> 4) << 24);
  static_assert(STAGE_BYTES % 1024 == 0, "stages stay 1024-byte aligned for the 128-byte swizzle");
};

// TMA loads into this CTA's shared memory that complete on a barrier of either
// CTA of the pair (`bar`: shared::cluster address).
__device__ __forceinline__ void tma2_load_3d(uint32_t dst, const void* tmap, uint32_t bar, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%3, %4, %5}], [%2];"
      :: "r"(dst), "l"(tmap), "r"(bar), "r"(x), "r"(y), "r"(z) : "memory");
}
__device__ __forceinline__ void tma2_load_4d(uint32_t dst, const void* tmap, uint32_t bar, int x, int y, int z,
                                             int w) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];"
      :: "r"(dst), "l"(tmap), "r"(bar), "r"(x), "r"(y), "r"(z), "r"(w) : "memory");
}
__device__ __forceinline__ void tc2_cp_sf(uint32_t tmem, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" :: "r"(tmem), "l"(sdesc) : "memory");
}
template <int MODE>
__device__ __forceinline__ void tc2_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                        uint32_t sfb, uint32_t accumulate) {
  if (MODE == 2) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
        :: "r"(d), "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate) : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
        :: "r"(d), "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate) : "memory");
  }
}

// (launched with a cluster dimension of 2; FQ: the fused call's quantize
// prologue first, in a cooperative launch)
template <int MODE, bool FQ>
__global__ void __launch_bounds__(kThreads, 1) qqmm_pair_kernel(
    const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
    const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
    const __grid_constant__ CUtensorMap tmO, const float* __restrict__ gs_x, const float* __restrict__ gs_w, int M,
    int N, int K, Batch bt, unsigned* __restrict__ err, int inject_timeout, FusedX fx) {
  using P = PairCfg<MODE>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  // per stage: [x rows | W rows | SFA | SFB rows 0-127 | SFB rows 128-255]; then
  // the epilogue warps' output staging (4 KB each); then the barriers
  uint8_t* stage_out = smem + kPairStages * P::STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(stage_out + kEpiWarps * 4096);
  uint64_t* full = bars;                       // CTA 0's are used
  uint64_t* empty = bars + kPairStages;
  uint64_t* acc_full = bars + 2 * kPairStages;
  uint64_t* acc_empty = bars + 2 * kPairStages + 1;  // CTA 0's is used
  uint64_t* never = bars + 2 * kPairStages + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kPairStages + 3);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int pair = (int)(blockIdx.x >> 1), npairs = (int)(gridDim.x >> 1);
  const int num_kb = K / BK;
  const int num_mp = (M + 255) / 256, num_n = (N + BN - 1) / BN;
  const int tiles_per_batch = num_mp * num_n;
  const int num_tiles = tiles_per_batch * bt.count;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPairStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 2 * kEpiWarps);
    mbar_init(never, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(tmem_slot)), "r"(TMEM_COLS) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  cluster_sync_all();  // both CTAs' barriers initialised and tensor memory allocated
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool failed = false;
  // programmatic dependent launch: the set-up above overlapped the previous
  // kernel's tail; x, its scales and the global scales may come from it
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (FQ)  // x -> codes and tiled scales in the workspace, through the idle operand ring
    quantize_prologue<MODE>(fx, M, K, smem, kPairStages * P::STAGE_BYTES, err, failed);

  if (warp == 0) {
    // ------------------------------------------------------------ producer --
    if (elect_one_sync()) {
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmB);
      prefetch_tmap(&tmSA);
      prefetch_tmap(&tmSB);
      int g = 0;
      for (int tile = pair; tile < num_tiles; tile += npairs) {
        const int b = tile / tiles_per_batch, rem = tile - b * tiles_per_batch;
        const int mp = rem % num_mp, n_blk = rem / num_mp;
        const int arow = mp * 256 + 128 * (int)rank;     // this CTA's x rows
        const int brow = n_blk * BN + 128 * (int)rank;   // this CTA's half of the W rows
        for (int kb = 0; kb < num_kb; ++kb, ++g) {
          const int s = g % kPairStages;
          const int round = g / kPairStages;
          if (round > 0) mbar_wait(&empty[s], (round - 1) & 1, err, failed);
          const uint32_t st = base + s * P::STAGE_BYTES;
          const uint32_t fb = mapa_u32(smem_u32(&full[s]), 0);
          if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * P::TX_CTA);
          tma2_load_3d(st, &tmA, fb, kb * BK_BYTES, arow, b);
          tma2_load_3d(st + A_BYTES, &tmB, fb, kb * BK_BYTES, brow, b * bt.wz);
          const int ty = kb * 2 * P::TPS;  // 256-byte rows of the scale view
          tma2_load_4d(st + P::AB_BYTES, &tmSA, fb, 0, ty, mp * 2 + (int)rank, b);
          tma2_load_4d(st + P::AB_BYTES + P::SF_BYTES, &tmSB, fb, 0, ty, n_blk * 2, b * bt.wz);
          tma2_load_4d(st + P::AB_BYTES + 2 * P::SF_BYTES, &tmSB, fb, 0, ty, n_blk * 2 + 1, b * bt.wz);
        }
      }
      // drain (CTA 0 sees both CTAs' fills): nothing may land after the pair
      // retires, so these waits run (bounded) even after an earlier one expired
      if (rank == 0) {
        bool drain_failed = false;
        for (int k = (g > kPairStages ? g - kPairStages : 0); k < g; ++k)
          mbar_wait_cluster(&full[k % kPairStages], (k / kPairStages) & 1, err, drain_failed);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------- MMA issuer (CTA 0) --
    if (rank == 0 && elect_one_sync()) {
      if (inject_timeout) {
        bool injected = false;
        mbar_wait(never, 0, err, injected, 2000000LL);
      }
      int g = 0, it = 0;
      for (int tile = pair; tile < num_tiles; tile += npairs, ++it) {
        if (it > 0) mbar_wait_cluster(acc_empty, (it - 1) & 1, err, failed);
        tc_fence_after();
        for (int kb = 0; kb < num_kb; ++kb, ++g) {
          const int s = g % kPairStages;
          mbar_wait_cluster(&full[s], (g / kPairStages) & 1, err, failed);
          tc_fence_after();
          const uint32_t st = base + s * P::STAGE_BYTES;
          const uint32_t sfa_smem = st + P::AB_BYTES;
          const uint32_t sfb_smem = sfa_smem + P::SF_BYTES;
          const uint32_t sfa_t = tmem + SF_COL + s * 48;
          const uint32_t sfb_t = sfa_t + 16;
#pragma unroll
          for (int j = 0; j < P::TPS; ++j) {
            tc2_cp_sf(sfa_t + 4 * j, desc_sf(sfa_smem + 512 * j));
            tc2_cp_sf(sfb_t + 8 * j, desc_sf(sfb_smem + 512 * j));
            tc2_cp_sf(sfb_t + 8 * j + 4, desc_sf(sfb_smem + P::SF_BYTES + 512 * j));
          }
          const uint64_t adesc = desc_sw128(st);
          const uint64_t bdesc = desc_sw128(st + A_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 64; ++k) {
            const int tl = (MODE == 2) ? k : (k >> 1);
            const uint32_t sf_id = (MODE == 2) ? 0u : (uint32_t)((k & 1) * 2);
            const uint32_t idesc = P::IDESC | (sf_id << 29) | (sf_id << 4);
            tc2_mma<MODE>(tmem + ACC_COL, adesc + (uint64_t)(2 * k), bdesc + (uint64_t)(2 * k), idesc,
                          sfa_t + 4 * tl, sfb_t + 8 * tl, (kb > 0 || k > 0) ? 1u : 0u);
          }
          tc2_commit_both(&empty[s]);
        }
        tc2_commit_both(acc_full);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue --
    // Warp (q, h) drains lane quadrant q, columns [128 h, 128 h + 128), of this
    // CTA's accumulator, releases it, then writes the 32 x 128 bf16 result as
    // two 32 x 64 boxes through a 4 KB shared-memory stage (128-byte swizzled,
    // so the row-per-lane writes hit every bank) and TMA tensor stores, which
    // clip rows >= M and columns >= N.
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;
    const uint32_t acc_empty0 = mapa_u32(smem_u32(acc_empty), 0);
    uint8_t* my_out = stage_out + (warp - 2) * 4096;
    const uint32_t my_out_s = smem_u32(my_out);
    int it = 0;
    for (int tile = pair; tile < num_tiles; tile += npairs, ++it) {
      const int b = tile / tiles_per_batch, rem = tile - b * tiles_per_batch;
      const int mp = rem % num_mp, n_blk = rem / num_mp;
      // (a fused call's activation scale was written by this grid: read it coherently)
      const float gx = gs_x ? (FQ ? __ldcg(gs_x + b) : __ldg(gs_x + b)) : 1.0f;
      const float alpha = __fmul_rn(gx, gs_w ? __ldg(gs_w + b) : 1.0f);
      mbar_wait(acc_full, it & 1, err, failed);
      tc_fence_after();
      // all 128 columns in flight at once, then the accumulator goes back to the MMAs
      uint32_t r[128];
      tmem_ld64(tmem + ((uint32_t)(32 * q) << 16) + ACC_COL + h * 128, r);
      tmem_ld64(tmem + ((uint32_t)(32 * q) << 16) + ACC_COL + h * 128 + 64, r + 64);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      // (the loads have completed: the signal publishes no memory, so no release)
      if (lane == 0) mbar_arrive_cluster_relaxed(acc_empty0);
      uint32_t o[64];
#pragma unroll
      for (int e = 0; e < 64; ++e)
        o[e] = pack_bf16x2_rn(__fmul_rn(__uint_as_float(r[2 * e]), alpha), __fmul_rn(__uint_as_float(r[2 * e + 1]), alpha));
      const int row0 = mp * 256 + 128 * (int)rank + 32 * q;
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {
        // the previous box's store has finished reading the stage
        if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4*>(my_out + lane * 128 + ((c ^ (lane & 7)) << 4)) =
              make_uint4(o[c2 * 32 + 4 * c], o[c2 * 32 + 4 * c + 1], o[c2 * 32 + 4 * c + 2], o[c2 * 32 + 4 * c + 3]);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        const int col0 = n_blk * BN + h * 128 + c2 * 64;
        if (lane == 0 && row0 < M && col0 < N) {  // (a box wholly outside the output is not issued)
          asm volatile(
              "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];"
              :: "l"(&tmO), "r"(col0), "r"(row0), "r"(b), "r"(my_out_s) : "memory");
          asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        }
      }
    }
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  }
  // no CTA of the pair retires while the other may still arrive on its barriers
  // or (CTA 0's MMAs) write its tensor memory
  tc_fence_before();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(TMEM_COLS) : "memory");
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

// 3-D map over packed codes viewed as bytes: [batch, rows, K/2] with the batch
// pitch in bytes, box 128 bytes x box_rows x 1.
bool make_code_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t K, uint32_t box_rows, int64_t batch,
                   int64_t batch_pitch) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)(K / 2), (cuuint64_t)rows, (cuuint64_t)batch};
  cuuint64_t strides[2] = {(cuuint64_t)(K / 2), (cuuint64_t)(batch > 1 ? batch_pitch : rows * (K / 2))};
  cuuint32_t box[3] = {(cuuint32_t)BK_BYTES, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int MODE>
cudaError_t launch_mode(const DevInfo& d, const uint32_t* xq, const uint8_t* sx, const uint32_t* wq,
                        const uint8_t* sw, const float* gs_x, const float* gs_w, int64_t M, int64_t N,
                        int64_t K, const BatchArgs& ba, uint16_t* out, int inject, cudaStream_t s) {
  CUtensorMap ta, tb;
  const bool shared_w = ba.stride_wq == 0;
  if (!make_code_map(&ta, xq, M, K, BM, ba.batch, ba.stride_xq * 4) ||
      !make_code_map(&tb, wq, N, K, BN, shared_w ? 1 : ba.batch, ba.stride_wq * 4))
    return cudaErrorInvalidValue;
  const size_t smem = Cfg<MODE>::SMEM_BYTES;
  if (smem > d.smem_optin) return cudaErrorInvalidValue;
  cudaError_t e =
      cudaFuncSetAttribute(qqmm_kernel<MODE, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  Batch bt;
  bt.count = (int)ba.batch;
  bt.wz = shared_w ? 0 : 1;
  bt.stride_sx = ba.stride_sx;
  bt.stride_sw = ba.stride_sw;
  bt.stride_out = ba.stride_out;
  const int64_t tiles = ((N + BN - 1) / BN) * ((M + BM - 1) / BM) * ba.batch;
  dim3 grid((unsigned)std::min<int64_t>(tiles, d.sm_count));
  qqmm_kernel<MODE, false><<<grid, kThreads, smem, s>>>(ta, tb, sx, sw, gs_x, gs_w, (int)M, (int)N, (int)K, bt,
                                                         out, d.err, inject, FusedX{});
  return cudaGetLastError();
}

// 4-D view of 128x4-tiled scale bytes [batch][row tiles][K tiles * 2][256 bytes]:
// one box is the TILES_PER_STAGE consecutive 512-byte tiles of one stage.
bool make_scale_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t K, int group, int tps, int64_t batch,
                    int64_t batch_pitch) {
  auto fn = encode_fn();
  if (!fn) return false;
  const int64_t rowtiles = (rows + 127) / 128;
  const int64_t ktiles = (K / group) / 4;  // 128x4 tiles along K per row tile
  cuuint64_t dims[4] = {256, (cuuint64_t)(ktiles * 2), (cuuint64_t)rowtiles, (cuuint64_t)batch};
  cuuint64_t strides[3] = {256, (cuuint64_t)(ktiles * 512),
                           (cuuint64_t)(batch > 1 ? batch_pitch : rowtiles * ktiles * 512)};
  cuuint32_t box[4] = {256, (cuuint32_t)(2 * tps), 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// bf16 output [batch][M][N] (batch pitch in elements) for TMA stores of 32-row x
// 64-column boxes, 128-byte swizzled in shared memory.
bool make_out_map(CUtensorMap* m, void* ptr, int64_t M, int64_t N, int64_t batch, int64_t batch_pitch) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)N, (cuuint64_t)M, (cuuint64_t)batch};
  cuuint64_t strides[2] = {(cuuint64_t)N * 2, (cuuint64_t)(batch > 1 ? batch_pitch : M * N) * 2};
  cuuint32_t box[3] = {64, 32, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, ptr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Pairs of the pair kernel that can be resident at once (cached per device and
// format; 0 if the query fails).
template <int MODE>
int pair_clusters(const DevInfo& d) {
  static std::mutex mu;
  static int cache[64];
  static bool have[64];
  if (d.device < 0 || d.device >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (have[d.device]) return cache[d.device];
  int n = 0;
  const int smem = (int)PairCfg<MODE>::SMEM_BYTES;
  if (cudaFuncSetAttribute(qqmm_pair_kernel<MODE, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) ==
          cudaSuccess &&
      cudaFuncSetAttribute(qqmm_pair_kernel<MODE, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) ==
          cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * std::max(1, d.sm_count / 2)));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, qqmm_pair_kernel<MODE, false>, &cfg) != cudaSuccess) {
      n = 0;
      cudaGetLastError();
    }
  } else {
    cudaGetLastError();
  }
  cache[d.device] = n;
  have[d.device] = true;
  return n;
}

template <int MODE>
cudaError_t launch_pair_mode(const DevInfo& d, int npairs_max, const uint32_t* xq, const uint8_t* sx,
                             const uint32_t* wq, const uint8_t* sw, const float* gs_x, const float* gs_w, int64_t M,
                             int64_t N, int64_t K, const BatchArgs& ba, uint16_t* out, int inject, cudaStream_t s) {
  using P = PairCfg<MODE>;
  constexpr int group = MODE == 2 ? 16 : 32;
  CUtensorMap ta, tb, tsa, tsb, to;
  const bool shared_w = ba.stride_wq == 0;
  const int64_t wb = shared_w ? 1 : ba.batch;
  if (!make_code_map(&ta, xq, M, K, 128, ba.batch, ba.stride_xq * 4) ||
      !make_code_map(&tb, wq, N, K, 128, wb, ba.stride_wq * 4) ||
      !make_scale_map(&tsa, sx, M, K, group, P::TPS, ba.batch, ba.stride_sx) ||
      !make_scale_map(&tsb, sw, N, K, group, P::TPS, (shared_w || ba.stride_sw == 0) ? 1 : ba.batch, ba.stride_sw) ||
      !make_out_map(&to, out, M, N, ba.batch, ba.stride_out))
    return cudaErrorInvalidValue;
  Batch bt;
  bt.count = (int)ba.batch;
  bt.wz = shared_w ? 0 : 1;
  bt.stride_out = ba.stride_out;
  const int64_t tiles = ((N + BN - 1) / BN) * ((M + 255) / 256) * ba.batch;
  const int npairs = (int)std::min<int64_t>(tiles, npairs_max);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * npairs));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = P::SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, qqmm_pair_kernel<MODE, false>, ta, tb, tsa, tsb, to, gs_x, gs_w, (int)M, (int)N,
                            (int)K, bt, d.err, inject, FusedX{});
}

// Workspace of a fused call: [codes | tiled scales | per-CTA partial maxima |
// global scale | barrier words], each part 128-byte aligned.
struct FusedWs {
  size_t xq = 0, sx = 0, partials = 0, gs = 0, bar = 0, total = 0;
  int64_t padded_rows = 0, padded_cols = 0;
};

FusedWs fused_ws_layout(int64_t M, int64_t K, int mode) {
  FusedWs w;
  const int group = mode == 2 ? 16 : 32;
  w.padded_rows = (M + 127) / 128 * 128;
  w.padded_cols = ((K / group) + 3) / 4 * 4;
  auto up = [](size_t v) { return (v + 127) / 128 * 128; };
  w.xq = 0;
  w.sx = up((size_t)M * (size_t)K / 2);
  w.partials = w.sx + up((size_t)(w.padded_rows * w.padded_cols));
  w.gs = w.partials + 1024 * 4;
  w.bar = w.gs + 128;
  w.total = w.bar + 128;
  return w;
}

template <int MODE>
cudaError_t launch_fused_mode(const DevInfo& d, const uint16_t* x, const float* gs_in, float* gs_out,
                              const uint32_t* wq, const uint8_t* sw, const float* gs_w, int64_t M, int64_t N,
                              int64_t K, uint8_t* ws, uint16_t* out, int inject, cudaStream_t s) {
  const FusedWs L = fused_ws_layout(M, K, MODE);
  FusedX fx;
  fx.x = x;
  fx.gs_in = gs_in;
  fx.gs_out = MODE == 2 ? reinterpret_cast<float*>(ws + L.gs) : nullptr;
  fx.gs_user = MODE == 2 ? gs_out : nullptr;
  fx.xq = reinterpret_cast<uint32_t*>(ws + L.xq);
  fx.sx = ws + L.sx;
  fx.partials = reinterpret_cast<uint32_t*>(ws + L.partials);
  fx.bar = reinterpret_cast<unsigned*>(ws + L.bar);
  fx.padded_rows = (int)L.padded_rows;
  fx.padded_cols = (int)L.padded_cols;
  const int np = pair_clusters<MODE>(d);
  if (np > 0) {
    // the CTA-pair kernel, cooperative (every CTA resident for the prologue's grid
    // barriers) with clusters of two
    using P = PairCfg<MODE>;
    constexpr int group = MODE == 2 ? 16 : 32;
    CUtensorMap ta, tb, tsa, tsb, to;
    if (!make_code_map(&ta, fx.xq, M, K, 128, 1, 0) || !make_code_map(&tb, wq, N, K, 128, 1, 0) ||
        !make_scale_map(&tsa, fx.sx, M, K, group, P::TPS, 1, 0) ||
        !make_scale_map(&tsb, sw, N, K, group, P::TPS, 1, 0) || !make_out_map(&to, out, M, N, 1, 0))
      return cudaErrorInvalidValue;
    const int64_t tiles = ((N + BN - 1) / BN) * ((M + 255) / 256);
    const int npairs = (int)std::min<int64_t>(std::min<int64_t>(tiles, np), 512);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * npairs));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = P::SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, qqmm_pair_kernel<MODE, true>, ta, tb, tsa, tsb, to,
                              (const float*)(MODE == 2 ? fx.gs_out : nullptr), gs_w, (int)M, (int)N, (int)K,
                              Batch{}, d.err, inject, fx);
  }
  CUtensorMap ta, tb;
  if (!make_code_map(&ta, fx.xq, M, K, BM, 1, 0) || !make_code_map(&tb, wq, N, K, BN, 1, 0))
    return cudaErrorInvalidValue;
  const size_t smem = Cfg<MODE>::SMEM_BYTES;
  if (smem > d.smem_optin) return cudaErrorInvalidValue;
  cudaError_t e =
      cudaFuncSetAttribute(qqmm_kernel<MODE, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t tiles = ((N + BN - 1) / BN) * ((M + BM - 1) / BM);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)std::min<int64_t>(std::min<int64_t>(tiles, d.sm_count), 1024));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // the grid barriers need every CTA resident
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, qqmm_kernel<MODE, true>, ta, tb, (const uint8_t*)fx.sx, sw,
                         (const float*)(MODE == 2 ? fx.gs_out : nullptr), gs_w, (int)M, (int)N, (int)K, Batch{}, out,
                         d.err, inject, fx);
  return e;
}

}  // namespace

cudaError_t launch_qqmm(const DevInfo& d, const uint32_t* xq, const uint8_t* sx, const uint32_t* wq,
                        const uint8_t* sw, const float* gs_x, const float* gs_w, int64_t M,
                        int64_t N, int64_t K, const BatchArgs& ba, int mode, uint16_t* out, int inject_timeout,
                        cudaStream_t s) {
  // the CTA-pair kernel whenever pairs of it can be resident; the one-SM kernel otherwise
  const int np = mode == 2 ? pair_clusters<2>(d) : pair_clusters<1>(d);
  if (np > 0) {
    if (mode == 2) return launch_pair_mode<2>(d, np, xq, sx, wq, sw, gs_x, gs_w, M, N, K, ba, out, inject_timeout, s);
    return launch_pair_mode<1>(d, np, xq, sx, wq, sw, gs_x, gs_w, M, N, K, ba, out, inject_timeout, s);
  }
  if (mode == 2) return launch_mode<2>(d, xq, sx, wq, sw, gs_x, gs_w, M, N, K, ba, out, inject_timeout, s);
  return launch_mode<1>(d, xq, sx, wq, sw, gs_x, gs_w, M, N, K, ba, out, inject_timeout, s);
}

size_t qqmm_fused_workspace_bytes(int64_t M, int64_t K, int mode) { return fused_ws_layout(M, K, mode).total; }

cudaError_t launch_qqmm_fused(const DevInfo& d, const uint16_t* x, const float* gs_in, float* gs_out,
                              const uint32_t* wq, const uint8_t* sw, const float* gs_w, int64_t M, int64_t N,
                              int64_t K, int mode, void* ws, uint16_t* out, int inject_timeout, cudaStream_t s) {
  if (mode == 2)
    return launch_fused_mode<2>(d, x, gs_in, gs_out, wq, sw, gs_w, M, N, K, static_cast<uint8_t*>(ws), out,
                                inject_timeout, s);
  return launch_fused_mode<1>(d, x, nullptr, nullptr, wq, sw, nullptr, M, N, K, static_cast<uint8_t*>(ws), out,
                              inject_timeout, s);
}

}  // namespace fp4
