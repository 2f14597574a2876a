// gather_qmm.cu -- MoE grouped GEMM: bf16 activations x MXFP4 expert weights
// (W4A16) on the tensor cores.
//
// Pages: "epic: NVIDIA Volta (sm_70) inference acceleration program #1536"
// (Diagnosis 1: gather_gemm; Diagnosis 5: the MoE grouped GEMM); "mlx: opt-in
// dense GEMM for nvfp4 prefill ... - #287" (the mixed-input GEMM whose weights
// are dequantized by producer warps in shared memory before bf16 tensor-core
// MMAs).
//
// Design: rows arrive sorted by expert.  Each CTA owns one tile of up to 256
// rows of one expert's segment (tiles never straddle experts; the tile ->
// expert map is rebuilt in every CTA by binary searches over the sorted expert
// ids, so no workspace is needed) and one 256-column slice of N.  Per K = 64
// stage:
//   * 16 producer warps gather the tile's activation rows with cp.async (16
//     bytes per copy, written in the 128-byte-swizzled K-major layout) and
//     dequantize the 256 x 64 weight slice exactly to bf16 (e2m1 *
//     2^(byte-127)) into the same layout, once for both 128-row halves of the
//     tile; each thread's weight codes and scales are loaded kPD stages ahead
//     into registers;
//   * one thread issues tcgen05.mma.kind::f16 (bf16 x bf16, fp32 accumulators
//     in tensor memory, M 128, N 256, K 16 per instruction): one MMA per half
//     that holds rows, each into its own 256-column accumulator;
//   * after the last stage warps 0-7 (lane quadrant warp % 4, half warp / 4)
//     read the accumulators (tcgen05.ld) and store bf16 rows of `out` in
//     routed-row order.
#include <algorithm>

#include "common.cuh"
#include "launch.h"

namespace fp4 {

namespace {

constexpr int BM = 128;                // rows per MMA (one accumulator)
constexpr int TM = 2 * BM;             // rows per tile: two MMA halves share each weight slice
constexpr int BN = 256;
constexpr int BK = 64;                 // bf16 elements per stage row: 128 bytes
constexpr int STAGES = 3;
constexpr int kProducerWarps = 16;
constexpr int kPD = 2;                 // weight prefetch distance (stages) in the producers' registers
constexpr int kProducers = kProducerWarps * 32;
constexpr int kThreads = kProducers + 32;  // + MMA warp
constexpr uint32_t A_HALF = BM * BK * 2;   // 16 KB: one 128-row half of the activations
constexpr uint32_t A_BYTES = 2 * A_HALF;   // 32 KB
constexpr uint32_t B_BYTES = BN * BK * 2;  // 32 KB
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 2048;
constexpr uint32_t TMEM_COLS = 512;        // accumulator of half h at column 256 h
// kind::f16 instruction descriptor: fp32 accumulator, bf16 A and B, K-major, N>>3, M>>4
constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                           ((uint32_t)(BM >> 4) << 24);

__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// byte offset of 16-byte chunk `c` (0..7) of row `r` in a 128-byte-swizzled tile
__device__ __forceinline__ uint32_t sw128(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" :: "r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

__global__ void __launch_bounds__(kThreads, 1) gather_qmm_kernel(
    const uint16_t* __restrict__ x, const int32_t* __restrict__ lhs, const int32_t* __restrict__ rhs,
    int R, const uint32_t* __restrict__ w, const uint8_t* __restrict__ scales, int E, int N, int K,
    uint16_t* __restrict__ out, unsigned* __restrict__ err, int inject_timeout) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* accum_full = bars + 2 * STAGES;
  uint64_t* never = bars + 2 * STAGES + 1;  // fault injection: a barrier nothing arrives at
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 2);
  int* tile_info = reinterpret_cast<int*>(bars + 2 * STAGES + 3);  // expert, row0, rows
  int* row_src = tile_info + 4;                                     // TM activation rows

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * BN;
  const int tile_id = blockIdx.y;

  // ---- tile -> (expert, first routed row, row count) --------------------
  if (warp == 0) {
    int prefix = 0, found = 0, fe = 0, frow = 0, frows = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      int lo_b = 0, hi_b = 0;
      if (e < E) {
        int lo = 0, hi = R;  // first index with rhs >= e
        while (lo < hi) { const int mid = (lo + hi) >> 1; if (__ldg(rhs + mid) < e) lo = mid + 1; else hi = mid; }
        lo_b = lo;
        lo = lo_b; hi = R;   // first index with rhs >= e + 1
        while (lo < hi) { const int mid = (lo + hi) >> 1; if (__ldg(rhs + mid) < e + 1) lo = mid + 1; else hi = mid; }
        hi_b = lo;
      }
      const int tiles = (hi_b - lo_b + TM - 1) / TM;
      int incl = tiles;
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      const int excl = prefix + incl - tiles;
      const bool mine = !found && tiles > 0 && tile_id >= excl && tile_id < excl + tiles;
      const unsigned hit = __ballot_sync(0xffffffffu, mine);
      if (hit) {
        const int src = __ffs(hit) - 1;
        const int r0 = lo_b + (tile_id - excl) * TM;
        const int re = __shfl_sync(0xffffffffu, r0, src);
        const int rend = __shfl_sync(0xffffffffu, hi_b, src);
        fe = e0 + src;
        frow = re;
        frows = min(TM, rend - re);
        found = 1;
      }
      prefix += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      tile_info[0] = found ? fe : -1;
      tile_info[1] = frow;
      tile_info[2] = frows;
    }
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], kProducers);
      mbar_init(&empty[s], 1);
    }
    mbar_init(accum_full, 1);
    mbar_init(never, 1);
    fence_barrier_init();
  }
  // The first CTA checks the routing contract once: every expert id in [0, E)
  // and non-decreasing.  A row outside it gets no tile (its output row is not
  // written); the error word reports it as an invalid argument.
  if (blockIdx.x == 0 && blockIdx.y == 0) {
    bool bad = false;
    for (int i = threadIdx.x; i < R; i += blockDim.x) {
      const int e = __ldg(rhs + i);
      bad |= e < 0 || e >= E || (i + 1 < R && e > __ldg(rhs + i + 1));
    }
    if (__syncthreads_or(bad) && threadIdx.x == 0) record_error(err, kErrIndex);
  }
  __syncthreads();
  const int expert = tile_info[0];
  if (expert < 0) return;  // uniform: this grid slot has no tile
  const int row0 = tile_info[1], rows = tile_info[2];
  for (int r = threadIdx.x; r < TM; r += blockDim.x) row_src[r] = (r < rows) ? __ldg(lhs + row0 + r) : 0;
  const int halves = rows > BM ? 2 : 1;  // 128-row halves holding rows (uniform)
  if (warp == kProducerWarps) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(tmem_slot)), "r"(TMEM_COLS) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;
  const int num_kb = K / BK;
  bool failed = false;  // this thread gave up a wait (see mbar_wait)

  if (warp < kProducerWarps) {
    // ---------------------------------------------------------- producers --
    const int t = threadIdx.x;
    const int64_t words_per_row = K / 8;
    const int64_t groups_per_row = K / 32;
    const uint32_t* we = w + (int64_t)expert * N * words_per_row;
    const uint8_t* se = scales + (int64_t)expert * N * groups_per_row;
    // Each thread dequantizes kItems (row, 32-code group) items per stage.  Their
    // codes and scales are loaded kPD stages ahead into a register ring, so the
    // global-memory latency overlaps the dequantization of the stages between.
    constexpr int kItems = (BN * 2) / kProducers;
    uint4 qr[kPD + 1][kItems];
    uint32_t sr[kPD + 1][kItems];
    auto load_w = [&](int kb, uint4 (&q)[kItems], uint32_t (&sc)[kItems]) {
#pragma unroll
      for (int i = 0; i < kItems; ++i) {
        const int item = t + kProducers * i;
        const int n = item >> 1, g = item & 1;
        if (n0 + n < N) {
          q[i] = ld_stream_v4(we + (int64_t)(n0 + n) * words_per_row + (kb * BK + g * 32) / 8);
          sc[i] = __ldg(se + (int64_t)(n0 + n) * groups_per_row + kb * 2 + g);
        } else {
          q[i] = make_uint4(0, 0, 0, 0);
          sc[i] = 0;
        }
      }
    };
#pragma unroll
    for (int u = 0; u < kPD; ++u)
      if (u < num_kb) load_w(u, qr[u], sr[u]);
    for (int kb0 = 0; kb0 < num_kb; kb0 += kPD + 1) {
#pragma unroll
      for (int u = 0; u <= kPD; ++u) {
        const int kb = kb0 + u;
        if (kb < num_kb) {
          if (kb + kPD < num_kb) load_w(kb + kPD, qr[(u + kPD) % (kPD + 1)], sr[(u + kPD) % (kPD + 1)]);
          const int s = kb % STAGES;
          const int round = kb / STAGES;
          if (round > 0) mbar_wait(&empty[s], (round - 1) & 1, err, failed);
          const uint32_t a_s = base + s * STAGE_BYTES;
          uint8_t* b_s = smem + s * STAGE_BYTES + A_BYTES;
          // activations: up to 256 rows x 8 chunks of 16 bytes (half h at A_HALF h;
          // a second half with no rows is not copied, its MMA is not issued)
#pragma unroll
          for (int i = 0; i < (TM * 8) / kProducers; ++i) {
            const int idx = t + kProducers * i;
            const int r = idx >> 3, c = idx & 7;
            if (r < BM * halves) {
              const uint16_t* src = x + (int64_t)row_src[r] * K + kb * BK + c * 8;
              cp_async16(a_s + sw128(r, c), src, r < rows ? 16u : 0u);
            }
          }
          asm volatile("cp.async.commit_group;" ::: "memory");
          // weights: 256 rows x 2 groups of 32 codes, dequantized to bf16 (exact)
#pragma unroll
          for (int i = 0; i < kItems; ++i) {
            const int item = t + kProducers * i;
            const int n = item >> 1, g = item & 1;
            const float sc = e8m0_to_f32(sr[u][i]);
            const uint32_t wv[4] = {qr[u][i].x, qr[u][i].y, qr[u][i].z, qr[u][i].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              uint32_t pk[4];
#pragma unroll
              for (int bb = 0; bb < 4; ++bb) {
                const uint32_t h2 = e2m1x2_to_f16x2((wv[j] >> (8 * bb)) & 0xFFu);
                pk[bb] = pack_bf16x2_rn(__fmul_rn(f16_lo_to_f32(h2), sc), __fmul_rn(f16_hi_to_f32(h2), sc));
              }
              *reinterpret_cast<uint4*>(b_s + sw128(n, g * 4 + j)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
          }
          // stage kb-1 is complete once its copies landed: publish it
          if (kb > 0) {
            asm volatile("cp.async.wait_group 1;" ::: "memory");
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_arrive(&full[(kb - 1) % STAGES]);
          }
        }
      }
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    mbar_arrive(&full[(num_kb - 1) % STAGES]);
  } else {
    // ------------------------------------------------------------ MMA warp --
    if (elect_one_sync()) {
      if (inject_timeout) {
        bool injected = false;  // separate flag: the injected expiry must not stop later waits
        mbar_wait(never, 0, err, injected, 2000000LL);
      }
      for (int kb = 0; kb < num_kb; ++kb) {
        const int s = kb % STAGES;
        mbar_wait(&full[s], (kb / STAGES) & 1, err, failed);
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint64_t adesc = desc_sw128(base + s * STAGE_BYTES);
        const uint64_t bdesc = desc_sw128(base + s * STAGE_BYTES + A_BYTES);
#pragma unroll
        for (int k = 0; k < BK / 16; ++k) {
          const uint32_t acc = (kb > 0 || k > 0) ? 1u : 0u;
          for (int hh = 0; hh < halves; ++hh)  // half hh: its 128 rows (16 KB further), its accumulator
            asm volatile(
                "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
                "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                :: "r"(tmem + 256u * hh), "l"(adesc + (uint64_t)(2 * k + (A_HALF >> 4) * hh)),
                   "l"(bdesc + (uint64_t)(2 * k)), "r"(IDESC), "r"(acc)
                : "memory");
        }
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                     :: "r"(smem_u32(&empty[s])) : "memory");
      }
      asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                   :: "r"(smem_u32(accum_full)) : "memory");
    }
  }

  // -------------------------------------------------------------- epilogue --
  if (warp < 4 * halves) {
    mbar_wait(accum_full, 0, err, failed);
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const int q = warp & 3, hh = warp >> 2;  // lane quadrant, half
    const int r = BM * hh + 32 * q + lane;
    uint16_t* orow = out + (int64_t)(row0 + r) * N;
#pragma unroll 1
    for (int c = 0; c < BN; c += 16) {
      uint32_t v[16];
      asm volatile(
          "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
          : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
            "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
          : "r"(tmem + ((uint32_t)(32 * q) << 16) + 256u * hh + c));
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
      const int col = n0 + c;
      if (r < rows) {
        uint4 o0, o1;
        o0.x = pack_bf16x2_rn(__uint_as_float(v[0]), __uint_as_float(v[1]));
        o0.y = pack_bf16x2_rn(__uint_as_float(v[2]), __uint_as_float(v[3]));
        o0.z = pack_bf16x2_rn(__uint_as_float(v[4]), __uint_as_float(v[5]));
        o0.w = pack_bf16x2_rn(__uint_as_float(v[6]), __uint_as_float(v[7]));
        o1.x = pack_bf16x2_rn(__uint_as_float(v[8]), __uint_as_float(v[9]));
        o1.y = pack_bf16x2_rn(__uint_as_float(v[10]), __uint_as_float(v[11]));
        o1.z = pack_bf16x2_rn(__uint_as_float(v[12]), __uint_as_float(v[13]));
        o1.w = pack_bf16x2_rn(__uint_as_float(v[14]), __uint_as_float(v[15]));
        if (col < N) *reinterpret_cast<uint4*>(orow + col) = o0;
        if (col + 8 < N) *reinterpret_cast<uint4*>(orow + col + 8) = o1;
      }
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == kProducerWarps) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(TMEM_COLS) : "memory");
  }
}

}  // namespace

cudaError_t launch_gather_qmm(const DevInfo& d, const uint16_t* x, const int32_t* lhs,
                              const int32_t* rhs, int64_t R, const uint32_t* w,
                              const uint8_t* scales, int64_t E, int64_t N, int64_t K, int mode,
                              uint16_t* out, int inject_timeout, cudaStream_t s) {
  (void)mode;
  if (SMEM_BYTES > d.smem_optin) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(gather_qmm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int64_t m_tiles = (R + TM - 1) / TM + E;  // upper bound on per-expert tiles
  dim3 grid((unsigned)((N + BN - 1) / BN), (unsigned)m_tiles);
  gather_qmm_kernel<<<grid, kThreads, SMEM_BYTES, s>>>(x, lhs, rhs, (int)R, w, scales, (int)E, (int)N,
                                                       (int)K, out, d.err, inject_timeout);
  return cudaGetLastError();
}

}  // namespace fp4
