// gather_qmm.cu -- 4-bit-weight x bf16-activation GEMMs on the tensor cores
// (W4A16): the MoE grouped GEMM gather_qmm and the dense prefill GEMM qmm, for
// MXFP4, NVFP4 and affine-4 weights.
//
// Pages: "epic: NVIDIA Volta (sm_70) inference acceleration program #1536"
// (Diagnosis 1: gather_gemm; Diagnosis 5: the MoE grouped GEMM); "mlx: opt-in
// dense GEMM for nvfp4 prefill ... - #287" (the mixed-input GEMM whose weights
// are dequantized by producer warps in shared memory before bf16 tensor-core
// MMAs, measured at 55-73 TFLOP/s for MLX's qmm and 285-324 TFLOP/s for the
// hand-written kernel on an RTX PRO 6000); "perf(cuda): enable hardware
// NVFP4/MXFP4 conversion on Blackwell builds" (qmm_sm80, the prefill qmm).
//
// Design.  A CTA owns one tile of up to 256 rows and one 256-column slice of N.
// gather_qmm: rows arrive sorted by expert; tiles never straddle experts (the
// tile -> expert map is rebuilt in every CTA from the expert ids, copied once
// into the still idle stage ring, so no workspace is needed).  qmm: the
// identity routing, one "expert", tile t = rows 256 t ...  Per K = 64 stage:
//   * 16 producer warps dequantize the 256 x 64 weight slice exactly to bf16
//     into the 128-byte-swizzled K-major layout the MMA reads, once for both
//     128-row halves of the tile; each thread's codes and scales are loaded kPD
//     stages ahead into registers.  MXFP4: e2m1 * 2^(byte - 127); NVFP4: e2m1 *
//     E4M3 (both exact in bf16; the NVFP4 global scale is applied in fp32 in the
//     epilogue); affine: w = q * scale + bias in fp32 split into two bf16 terms
//     hi = bf16(w), lo = bf16(w - hi) (a single bf16 rounding of w would cost
//     ~2.5e-3 relative error), each its own B operand;
//   * activations: qmm loads one TMA box of 256 rows x 128 bytes per stage (rows
//     past M read as zeros); gather_qmm loads a tile whose routed rows are
//     consecutive rows of x by 128-row TMA boxes, and otherwise gathers rows
//     with cp.async (16 bytes per copy, written in the same swizzled layout),
//     the copies arriving on the stage barrier by themselves when they land;
//   * one thread issues tcgen05.mma.kind::f16 (bf16 x bf16, fp32 accumulators
//     in tensor memory, M 128, N 256, K 16 per instruction): per half that holds
//     rows one MMA (two for affine: hi then lo), each half into its own
//     256-column accumulator;
//   * after the last stage warps 0-7 (lane quadrant warp % 4, half warp / 4)
//     read the accumulators (tcgen05.ld) and write bf16 rows of `out` through a
//     swizzled shared-memory stage and TMA tensor stores.
// Every mbarrier wait is bounded (an expired wait records FP4_ERR_TIMEOUT).
#include <algorithm>
#include <mutex>
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "launch.h"
#include "pair.cuh"

namespace fp4 {

namespace {

constexpr int BM = 128;                // rows per MMA (one accumulator)
constexpr int BK = 64;                 // bf16 elements per stage row: 128 bytes
constexpr int kProducerWarps = 16;
constexpr int kPD = 2;                 // weight prefetch distance (stages) in the producers' registers
constexpr int kProducers = kProducerWarps * 32;
constexpr int kThreads = kProducers + 32;  // + MMA warp
constexpr uint32_t A_HALF = BM * BK * 2;   // 16 KB: one 128-row half of the activations
constexpr uint32_t TMEM_COLS = 512;

// Tile geometry (qmm and gather_qmm): 256 rows (two 128-row MMA halves) x 256
// columns.  Measured on the MoE shapes against 384 x 160 (three halves, so that
// an expert of up to 384 rows is one tile) and 512 x 128: the N = 256 MMA is the
// fastest per flop by a wide margin, which outweighs dequantizing the weight
// slice again for an expert's last few rows.
constexpr int TM = 2 * BM;                 // rows per tile
constexpr int BN = 256;                    // columns per tile
constexpr uint32_t A_BYTES = 2 * A_HALF;   // 32 KB
constexpr uint32_t B_BYTES = BN * BK * 2;  // 32 KB per weight term
constexpr int kItems = 2 * BN;             // (row, 32-code half) items per stage: one per producer thread
static_assert(kItems == kProducers, "one weight item per producer thread per stage");
// kind::f16 instruction descriptor: fp32 accumulator, bf16 A and B, K-major, N>>3, M>>4
constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                           ((uint32_t)(BM >> 4) << 24);

// MODE 0 (affine) carries two weight terms per stage and fits two stages; the
// FP4 formats one term and three stages.
template <int MODE, bool DENSE> struct Cfg {
  static constexpr int kTerms = MODE == 0 ? 2 : 1;
  static constexpr int kStages = MODE == 0 ? 2 : 3;
  static constexpr uint32_t kStageBytes = A_BYTES + kTerms * B_BYTES;
  // + 1024 alignment slack, 256 for barriers and the tile info, and gather_qmm's
  // row map -- kept tight: past 196 KB per block the L1 that serves the weight
  // scale loads shrinks from 60 to 28 KB, which costs qmm ~20 %
  static constexpr uint32_t kReserve = 1024 + 256 + (DENSE ? 0 : TM * 4);
  static constexpr uint32_t kSmemBytes = kStages * kStageBytes + kReserve;
  static_assert(kStageBytes % 1024 == 0, "stages stay 1024-byte aligned for the 128-byte swizzle");
};

__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" :: "r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

// 32 lanes x 64 consecutive 32-bit tensor-memory columns (one register per column)
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

// byte offset of 16-byte chunk `c` (0..7) of row `r` in a 128-byte-swizzled tile
__device__ __forceinline__ uint32_t sw128(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

// The weight scale data of one (row, 32-code) item: MXFP4 one E8M0 byte, NVFP4
// two E4M3 bytes (16 codes each), affine the bf16 scale and bias packed.
template <int MODE>
__device__ __forceinline__ uint32_t load_item_scale(const void* scales, const uint16_t* biases, int64_t row,
                                                    int64_t K, int group, int64_t k0) {
  if (MODE == 1) return __ldg(static_cast<const uint8_t*>(scales) + row * (K / 32) + k0 / 32);
  if (MODE == 2) return __ldg(reinterpret_cast<const uint16_t*>(static_cast<const uint8_t*>(scales) + row * (K / 16) + k0 / 16));
  const int64_t gi = row * (K / group) + k0 / group;
  return (uint32_t)__ldg(static_cast<const uint16_t*>(scales) + gi) | ((uint32_t)__ldg(biases + gi) << 16);
}

// Dequantize one item (NW words: 8 NW codes of row n, item g of the stage row)
// into its NW swizzled 16-byte chunks of each term.
template <int MODE, int NW = 4>
__device__ __forceinline__ void dequant_item(uint4 q, uint32_t sc, uint8_t* b_hi, uint8_t* b_lo, int n, int g) {
  const uint32_t wv[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int j = 0; j < NW; ++j) {
    uint32_t hi[4], lo[4];
    if (MODE == 0) {
      const float s = bf16_lo(sc), b = bf16_hi(sc);
#pragma unroll
      for (int bb = 0; bb < 4; ++bb) {
        const uint32_t byte = (wv[j] >> (8 * bb)) & 0xFFu;
        // q via the 2^23 magic: exact small integers
        const float q0 = __fsub_rn(__uint_as_float(0x4B000000u | (byte & 15u)), 8388608.0f);
        const float q1 = __fsub_rn(__uint_as_float(0x4B000000u | (byte >> 4)), 8388608.0f);
        const float w0 = __fmaf_rn(q0, s, b), w1 = __fmaf_rn(q1, s, b);
        const uint32_t h = pack_bf16x2_rn(w0, w1);
        hi[bb] = h;
        lo[bb] = pack_bf16x2_rn(__fsub_rn(w0, bf16_lo(h)), __fsub_rn(w1, bf16_hi(h)));
      }
    } else {
      // NVFP4: word j holds codes 8j .. 8j + 7, scale byte (8j) / 16 = j / 2
      const float scale = (MODE == 1) ? e8m0_to_f32(sc) : e4m3_to_f32((sc >> (8 * (j >> 1))) & 0xFFu);
#pragma unroll
      for (int bb = 0; bb < 4; ++bb) {
        const uint32_t h2 = e2m1x2_to_f16x2((wv[j] >> (8 * bb)) & 0xFFu);
        hi[bb] = pack_bf16x2_rn(__fmul_rn(f16_lo_to_f32(h2), scale), __fmul_rn(f16_hi_to_f32(h2), scale));
      }
    }
    *reinterpret_cast<uint4*>(b_hi + sw128(n, g * NW + j)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    if (MODE == 0) *reinterpret_cast<uint4*>(b_lo + sw128(n, g * NW + j)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  }
}

template <int MODE, bool DENSE>
__global__ void __launch_bounds__(kThreads, 1) w4a16_kernel(
    const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmO,
    const uint16_t* __restrict__ x, const int32_t* __restrict__ lhs,
    const int32_t* __restrict__ rhs, int R, const uint32_t* __restrict__ w, const void* __restrict__ scales,
    const uint16_t* __restrict__ biases, const float* __restrict__ gs_w, int E, int N, int K, int group,
    uint16_t* __restrict__ out, unsigned* __restrict__ err, int inject_timeout) {
  using C = Cfg<MODE, DENSE>;
  constexpr int STAGES = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * C::kStageBytes);
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
  if (DENSE) {
    if (threadIdx.x == 0) {
      tile_info[0] = 0;
      tile_info[1] = tile_id * TM;
      tile_info[2] = min(TM, R - tile_id * TM);
    }
  }
  // The segment starts start[e] (first routed row whose id is >= e, e in [0, E]):
  // while the ids fit in the idle stage ring, one coalesced pass copies them to
  // shared memory and each row boundary fills the starts it separates (ids are
  // clamped to [-1, E], so a broken contract cannot index outside start[]);
  // otherwise warp 0 binary-searches global memory per expert.
  const bool smem_map = !DENSE && (int64_t)R + E + 1 <= (int64_t)(C::kStages * C::kStageBytes / 4);
  int* seg_start = reinterpret_cast<int*>(smem) + R;
  if (smem_map) {
    int* ids = reinterpret_cast<int*>(smem);
#pragma unroll 8
    for (int i = threadIdx.x; i < R; i += blockDim.x) {  // (unrolled: the loads overlap)
      const int e = __ldg(rhs + i);
      ids[i] = e < 0 ? -1 : min(e, E);
    }
    __syncthreads();
    for (int i = threadIdx.x; i <= R; i += blockDim.x) {
      const int prev = i > 0 ? ids[i - 1] : -1, cur = i < R ? ids[i] : E;
      for (int e = max(prev + 1, 0); e <= cur; ++e) seg_start[e] = i;
    }
    __syncthreads();
  }
  if (!DENSE && warp == 0) {
    int prefix = 0, found = 0, fe = 0, frow = 0, frows = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      int lo_b = 0, hi_b = 0;
      if (e < E && smem_map) {
        lo_b = seg_start[e];
        hi_b = max(seg_start[e + 1], lo_b);
      } else if (e < E) {
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
      // qmm: the producers' arrivals + the activation box's byte count; gather_qmm: the
      // producers' arrivals + one arrival per producer when its activation copies land
      mbar_init(&full[s], DENSE ? kProducers + 1 : 2 * kProducers);
      mbar_init(&empty[s], 1);
    }
    mbar_init(accum_full, 1);
    mbar_init(never, 1);
    fence_barrier_init();
  }
  // gather_qmm: the first CTA checks the routing contract once: every expert id
  // in [0, E) and non-decreasing.  A row outside it gets no tile (its output row
  // is not written); the error word reports it as an invalid argument.
  if (!DENSE && blockIdx.x == 0 && blockIdx.y == 0) {
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
  if (!DENSE)
    for (int r = threadIdx.x; r < TM; r += blockDim.x) row_src[r] = (r < rows) ? __ldg(lhs + row0 + r) : 0;
  const int halves = (rows + BM - 1) / BM;  // 128-row halves holding rows (uniform)
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
  // gather_qmm: a tile whose routed rows are consecutive rows of x (activations
  // already in routed order) loads its full 128-row halves by TMA boxes, like
  // qmm; a partial last half, and every half of a scattered tile, by cp.async
  int tma_halves = 0;
  if (!DENSE) {
    bool ok = true;
    for (int r = threadIdx.x; r < rows; r += blockDim.x) ok &= row_src[r] == row_src[0] + r;
    tma_halves = __syncthreads_and(ok) ? rows / BM : 0;
  }

  if (warp < kProducerWarps) {
    // ---------------------------------------------------------- producers --
    const int t = threadIdx.x;
    const int64_t words_per_row = K / 8;
    const int64_t erow0 = (int64_t)expert * N;  // first weight row of this expert
    const int n = t >> 1, g = t & 1;            // this thread's item: row n, codes 32 g .. 32 g + 31 of a stage
    const bool nrow_ok = n0 + n < N;
    const uint32_t* wrow = w + (erow0 + n0 + n) * words_per_row;
    // gather_qmm: this thread's activation copies, fixed for the tile -- 16-byte
    // chunk t % 8 of rows t / 8 + 64 i (source pointer at K offset 0, swizzled
    // destination offset within a stage)
    constexpr int kCopies = (TM * 8) / kProducers;
    const uint16_t* cp_src[kCopies];
    uint32_t cp_dst[kCopies];
    int cp_row[kCopies];
#pragma unroll
    for (int i = 0; i < kCopies; ++i) {
      const int idx = t + kProducers * i;
      cp_row[i] = idx >> 3;
      cp_dst[i] = sw128(idx >> 3, idx & 7);
      cp_src[i] = DENSE ? x : x + (int64_t)row_src[idx >> 3] * K + (idx & 7) * 8;
    }
    // codes and scales of the item, kPD stages ahead in a register ring
    uint4 qr[kPD + 1];
    uint32_t sr[kPD + 1];
    auto load_w = [&](int kb, uint4& q, uint32_t& sc) {
      if (nrow_ok) {
        q = ld_stream_v4(wrow + (kb * BK + g * 32) / 8);
        sc = load_item_scale<MODE>(scales, biases, erow0 + n0 + n, K, group, (int64_t)kb * BK + g * 32);
      } else {
        q = make_uint4(0, 0, 0, 0);
        sc = 0;
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
          const uint32_t a_s = base + s * C::kStageBytes;
          uint8_t* b_s = smem + s * C::kStageBytes + A_BYTES;
          if (DENSE) {
            // activations: one TMA box of TM rows x 128 bytes (rows past the matrix read as zeros)
            if (t == 0) {
              mbar_arrive_expect_tx(&full[s], (uint32_t)A_BYTES);
              tma_load_2d(smem + s * C::kStageBytes, &tmX, &full[s], kb * BK, row0);
            }
          } else {
            // activations: up to 256 rows x 8 chunks of 16 bytes (half h at A_HALF h; a
            // half with no rows is not loaded, its MMA is not issued).  Halves below
            // tma_halves: one TMA box of 128 whole rows each, whose bytes thread 0
            // adds to the stage's expected transaction count (no arrival); the rest by
            // cp.async, every thread's copies arriving on the stage barrier by
            // themselves when they land (cp.async.mbarrier.arrive.noinc), so no
            // producer waits for them.
            if (t == 0 && tma_halves > 0) {
              asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;"
                           :: "r"(smem_u32(&full[s])), "r"((uint32_t)(tma_halves * A_HALF)) : "memory");
              for (int h = 0; h < tma_halves; ++h)
                tma_load_2d(smem + s * C::kStageBytes + h * A_HALF, &tmX, &full[s], kb * BK, row_src[0] + h * BM);
            }
            if (tma_halves < halves) {  // (uniform) rows left for the 16-byte copies
#pragma unroll
              for (int i = 0; i < kCopies; ++i)
                if (cp_row[i] >= BM * tma_halves && cp_row[i] < BM * halves)
                  cp_async16(a_s + cp_dst[i], cp_src[i] + kb * BK, cp_row[i] < rows ? 16u : 0u);
            }
            asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" :: "r"(smem_u32(&full[s])) : "memory");
          }
          // weights: 256 rows x 2 items of 32 codes, dequantized to bf16 (one or two terms)
          dequant_item<MODE>(qr[u], sr[u], b_s, b_s + B_BYTES, n, g);
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          mbar_arrive(&full[s]);
        }
      }
    }
    // no copy may still be in flight when the block retires (the MMA thread may
    // have given up): thread 0's TMA boxes land on the last stages' barriers,
    // waited for (bounded) even after an earlier wait expired
    if (t == 0) {
      bool drain_failed = false;
      for (int kb = max(0, num_kb - STAGES); kb < num_kb; ++kb)
        mbar_wait(&full[kb % STAGES], (kb / STAGES) & 1, err, drain_failed);
    }
    if (!DENSE) asm volatile("cp.async.wait_all;" ::: "memory");
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
        // the activation rows were written by cp.async (generic proxy) and observed
        // through the barrier: make them visible to the tensor core's async proxy
        if (!DENSE) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint64_t adesc = desc_sw128(base + s * C::kStageBytes);
        const uint64_t bdesc = desc_sw128(base + s * C::kStageBytes + A_BYTES);
#pragma unroll
        for (int k = 0; k < BK / 16; ++k) {
#pragma unroll
          for (int tt = 0; tt < C::kTerms; ++tt) {
            const uint32_t acc = (kb > 0 || k > 0 || tt > 0) ? 1u : 0u;
            for (int hh = 0; hh < halves; ++hh)  // half hh: its 128 rows (16 KB further), its accumulator
              asm volatile(
                  "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
                  "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                  :: "r"(tmem + (uint32_t)(BN * hh)), "l"(adesc + (uint64_t)(2 * k + (A_HALF >> 4) * hh)),
                     "l"(bdesc + (uint64_t)(2 * k + (B_BYTES >> 4) * tt)), "r"(IDESC), "r"(acc)
                  : "memory");
          }
        }
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                     :: "r"(smem_u32(&empty[s])) : "memory");
      }
      asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                   :: "r"(smem_u32(accum_full)) : "memory");
    }
  }

  // -------------------------------------------------------------- epilogue --
  // Warp (q, hh) owns rows BM hh + 32 q .. + 31 of the tile: 64 columns at a time
  // from tensor memory, times the NVFP4 global scale, rounded to bf16.  A band
  // whose 32 rows all belong to the tile leaves through a 4 KB shared-memory
  // stage (128-byte swizzled; the ring is idle once the last MMA completed)
  // and a TMA tensor store, which clips columns >= N; the tile's last, partial
  // band is stored row by row.
  if (warp < 4 * halves) {
    mbar_wait(accum_full, 0, err, failed);
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const float gsw = (MODE == 2 && gs_w) ? __ldg(gs_w) : 1.0f;
    const int q = warp & 3, hh = warp >> 2;  // lane quadrant, half
    const int rb = BM * hh + 32 * q;         // first row of the band
    const int r = rb + lane;
    const bool full_band = rb + 32 <= rows;
    uint8_t* stage_o = smem + warp * 8192;   // two 4 KB boxes per warp
    uint16_t* orow = out + (int64_t)(row0 + r) * N;
#pragma unroll 1
    for (int c = 0; c < BN; c += 64) {
      uint32_t v[64];
      tmem_ld64(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(BN * hh + c), v);
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
      uint32_t o[32];
#pragma unroll
      for (int e = 0; e < 32; ++e)
        o[e] = pack_bf16x2_rn(__fmul_rn(__uint_as_float(v[2 * e]), gsw), __fmul_rn(__uint_as_float(v[2 * e + 1]), gsw));
      const int col = n0 + c;
      if (full_band) {
        uint8_t* box = stage_o + ((c >> 6) & 1) * 4096;
        if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");  // this box's previous store read it
        __syncwarp();
#pragma unroll
        for (int k = 0; k < 8; ++k)
          *reinterpret_cast<uint4*>(box + lane * 128 + ((k ^ (lane & 7)) << 4)) =
              make_uint4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
          if (col < N)
            asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];"
                         :: "l"(&tmO), "r"(col), "r"(row0 + rb), "r"(smem_u32(box)) : "memory");
          // one group per box, empty past N, so that "at most one pending" above
          // always means this box's previous store has read it
          asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        }
      } else if (r < rows) {
#pragma unroll
        for (int k = 0; k < 8; ++k)
          if (col + 8 * k < N)
            *reinterpret_cast<uint4*>(orow + col + 8 * k) = make_uint4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
      }
    }
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == kProducerWarps) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(TMEM_COLS) : "memory");
  }
}

// ---------------------------------------------------------------------------
// qmm on CTA pairs (tcgen05 cta_group::2).  A cluster of two CTAs owns 512
// rows x 256 columns of the output.  CTA r holds rows 128 r .. 128 r + 127 and
// 256 + 128 r .. 256 + 128 r + 127 of the tile's activations (two TMA boxes per
// stage) and dequantizes W rows n0 + 128 r .. n0 + 128 r + 127 (16 codes per
// producer thread).  One thread of CTA 0 issues, per 16-element k-step and
// weight term, two kind::f16 MMAs of M 256 (rows 0-255 and 256-511 of the
// tile), each reading both CTAs' activation rows and both CTAs' halves of the
// weight slice.  Each CTA accumulates its 2 x 128 rows x 256 columns in its own
// tensor memory.  An SM so dequantizes half the weights the one-SM tile does
// for the same MMA work.  Both CTAs' activation boxes complete on CTA 0's
// stage barrier.  Producer warps arrive on their own CTA's barrier (a CTA-scope
// release, which does not wait for their weight loads in flight); CTA 1's idle
// MMA warp forwards each completed stage to CTA 0's barrier with one arrival
// whose release has CTA scope (the stage's operands are this CTA's own shared
// memory).  A cluster-scope release waits for the SM's global loads in flight:
// by every producer warp it halved the speed, and by the forwarder alone it
// still held NVFP4 to ~1370 TFLOP/s.  CTA 0's commits free a stage (and
// publish the accumulators) in both CTAs.
template <int MODE>
struct PairQ {
  static constexpr int kTerms = MODE == 0 ? 2 : 1;
  static constexpr uint32_t kA = 2 * A_HALF;           // two 128-row blocks of x: 32 KB
  static constexpr uint32_t kB = (BN / 2) * BK * 2;    // 128 W rows x 64 bf16: 16 KB per term
  static constexpr uint32_t kStageBytes = kA + kTerms * kB;
  static constexpr int kStages = MODE == 0 ? 3 : 4;    // 192 KB of stages: below the 196 KB carve-out
  static constexpr uint32_t kSmemBytes = kStages * kStageBytes + 1024 + 256;
  static constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                                    ((uint32_t)(256 >> 4) << 24);
  static_assert(kStageBytes % 1024 == 0, "stages stay 1024-byte aligned for the 128-byte swizzle");
};
constexpr int kPairRows = 512;  // output rows per CTA pair
constexpr int kPairPD = 2;      // weight prefetch distance (stages) of the pair kernel's producers (4: no faster)

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) qmm_pair_kernel(
    const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmO, int M,
    const uint32_t* __restrict__ w, const void* __restrict__ scales, const uint16_t* __restrict__ biases,
    const float* __restrict__ gs_w, int N, int K, int group, uint16_t* __restrict__ out,
    unsigned* __restrict__ err, int inject_timeout) {
  using P = PairQ<MODE>;
  constexpr int STAGES = P::kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * P::kStageBytes);
  uint64_t* full = bars;                     // CTA 0's are used
  uint64_t* empty = bars + STAGES;
  uint64_t* accum_full = bars + 2 * STAGES;
  uint64_t* never = bars + 2 * STAGES + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int n0 = (int)(blockIdx.x >> 1) * BN;
  const int prow0 = (int)blockIdx.y * kPairRows;
  const int num_kb = K / BK;
  bool failed = false;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      // CTA 0: its producer warps, the byte count and CTA 1's forwarded stage; CTA 1: its producer warps
      mbar_init(&full[s], rank == 0 ? kProducerWarps + 2 : kProducerWarps);
      mbar_init(&empty[s], 1);
    }
    mbar_init(accum_full, 1);
    mbar_init(never, 1);
    fence_barrier_init();
  }
  if (warp == kProducerWarps) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(tmem_slot)), "r"(TMEM_COLS) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  cluster_sync_all();  // both CTAs' barriers initialised and tensor memory allocated
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;

  if (warp < kProducerWarps) {
    // ---------------------------------------------------------- producers --
    const int t = threadIdx.x;
    const int n = t >> 2, g = t & 3;  // this thread's item: W row n of the CTA's 128, codes 16 g .. 16 g + 15
    const int64_t wr = (int64_t)n0 + 128 * (int64_t)rank + n;
    const bool nrow_ok = wr < N;
    const uint32_t* wrow = w + wr * (K / 8);
    const uint32_t full0 = mapa_u32(smem_u32(full), 0);  // CTA 0's stage barriers (8 bytes apart)
    uint2 qr[kPairPD + 1];
    uint32_t sr[kPairPD + 1];
    auto load_w = [&](int kb, uint2& q, uint32_t& sc) {
      if (nrow_ok) {
        const int64_t k0 = (int64_t)kb * BK + g * 16;
        q = __ldg(reinterpret_cast<const uint2*>(wrow + k0 / 8));
        sc = (MODE == 2) ? (uint32_t)__ldg(static_cast<const uint8_t*>(scales) + wr * (K / 16) + k0 / 16)
                         : load_item_scale<MODE>(scales, biases, wr, K, group, k0);
      } else {
        q = make_uint2(0u, 0u);
        sc = 0;
      }
    };
#pragma unroll
    for (int u = 0; u < kPairPD; ++u)
      if (u < num_kb) load_w(u, qr[u], sr[u]);
    for (int kb0 = 0; kb0 < num_kb; kb0 += kPairPD + 1) {
#pragma unroll
      for (int u = 0; u <= kPairPD; ++u) {
        const int kb = kb0 + u;
        if (kb < num_kb) {
          if (kb + kPairPD < num_kb) load_w(kb + kPairPD, qr[(u + kPairPD) % (kPairPD + 1)], sr[(u + kPairPD) % (kPairPD + 1)]);
          const int s = kb % STAGES, round = kb / STAGES;
          if (round > 0) mbar_wait(&empty[s], (round - 1) & 1, err, failed);
          const uint32_t a_s = base + s * P::kStageBytes;
          uint8_t* b_s = smem + s * P::kStageBytes + P::kA;
          if (t == 0) {
            // this CTA's two 128-row blocks of x (rows past M read as zeros), counted on CTA 0's barrier
            if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * P::kA);
            tma2_load_2d(a_s, &tmX, full0 + 8 * s, kb * BK, prow0 + 128 * (int)rank);
            tma2_load_2d(a_s + A_HALF, &tmX, full0 + 8 * s, kb * BK, prow0 + 256 + 128 * (int)rank);
          }
          dequant_item<MODE, 2>(make_uint4(qr[u].x, qr[u].y, 0u, 0u), sr[u], b_s, b_s + P::kB, n, g);
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) mbar_arrive(&full[s]);  // this CTA's barrier
        }
      }
    }
    // no TMA box of either CTA may still be landing when the pair retires: CTA 0's
    // stage barriers count both CTAs' bytes; waited for (bounded) even after an
    // earlier wait expired
    if (t == 0 && rank == 0) {
      bool drain_failed = false;
      for (int kb = max(0, num_kb - STAGES); kb < num_kb; ++kb)
        mbar_wait_cluster(&full[kb % STAGES], (kb / STAGES) & 1, err, drain_failed);
    }
  } else if (rank == 0) {
    // ------------------------------------------------- MMA issuer (CTA 0) --
    if (elect_one_sync()) {
      if (inject_timeout) {
        bool injected = false;  // separate flag: the injected expiry must not stop later waits
        mbar_wait(never, 0, err, injected, 2000000LL);
      }
      for (int kb = 0; kb < num_kb; ++kb) {
        const int s = kb % STAGES;
        mbar_wait_cluster(&full[s], (kb / STAGES) & 1, err, failed);
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint64_t adesc = desc_sw128(base + s * P::kStageBytes);
        const uint64_t bdesc = desc_sw128(base + s * P::kStageBytes + P::kA);
#pragma unroll
        for (int k = 0; k < BK / 16; ++k) {
#pragma unroll
          for (int tt = 0; tt < P::kTerms; ++tt) {
            const uint32_t acc = (kb > 0 || k > 0 || tt > 0) ? 1u : 0u;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)  // rows 256 hh .. 256 hh + 255 of the tile, accumulator hh
              asm volatile(
                  "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
                  "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                  :: "r"(tmem + (uint32_t)(BN * hh)), "l"(adesc + (uint64_t)(2 * k + (A_HALF >> 4) * hh)),
                     "l"(bdesc + (uint64_t)(2 * k + (P::kB >> 4) * tt)), "r"(P::IDESC), "r"(acc)
                  : "memory");
          }
        }
        tc2_commit_both(&empty[s]);
      }
      tc2_commit_both(accum_full);
    }
  } else {
    // ------------------------------------- CTA 1: forward completed stages --
    if (elect_one_sync()) {
      const uint32_t full0 = mapa_u32(smem_u32(full), 0);
      for (int kb = 0; kb < num_kb; ++kb) {
        const int s = kb % STAGES;
        mbar_wait(&full[s], (kb / STAGES) & 1, err, failed);
        mbar_arrive_remote_cta(full0 + 8 * s);
      }
    }
  }

  // -------------------------------------------------------------- epilogue --
  // Warp (q, hh) of either CTA owns rows row_base + 32 q .. + 31, row_base =
  // prow0 + 256 hh + 128 rank, of accumulator hh: as the one-SM kernel's
  // epilogue (full 32-row bands by TMA stores through a swizzled 4 KB stage,
  // the last partial band row by row).  The operand ring is idle in both CTAs
  // once the final commit has arrived.
  if (warp < 8) {
    mbar_wait(accum_full, 0, err, failed);
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const float gsw = (MODE == 2 && gs_w) ? __ldg(gs_w) : 1.0f;
    const int q = warp & 3, hh = warp >> 2;
    const int row_base = prow0 + 256 * hh + 128 * (int)rank;
    const int rows = max(0, min(128, M - row_base));
    const int rb = 32 * q;
    const int r = rb + lane;
    const bool full_band = rb + 32 <= rows;
    uint8_t* stage_o = smem + warp * 8192;
    uint16_t* orow = out + (int64_t)(row_base + r) * N;
#pragma unroll 1
    for (int c = 0; c < BN; c += 64) {
      uint32_t v[64];
      tmem_ld64(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(BN * hh + c), v);
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
      uint32_t o[32];
#pragma unroll
      for (int e = 0; e < 32; ++e)
        o[e] = pack_bf16x2_rn(__fmul_rn(__uint_as_float(v[2 * e]), gsw), __fmul_rn(__uint_as_float(v[2 * e + 1]), gsw));
      const int col = n0 + c;
      if (full_band) {
        uint8_t* box = stage_o + ((c >> 6) & 1) * 4096;
        if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
        __syncwarp();
#pragma unroll
        for (int k = 0; k < 8; ++k)
          *reinterpret_cast<uint4*>(box + lane * 128 + ((k ^ (lane & 7)) << 4)) =
              make_uint4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
          if (col < N)
            asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];"
                         :: "l"(&tmO), "r"(col), "r"(row_base + rb), "r"(smem_u32(box)) : "memory");
          asm volatile("cp.async.bulk.commit_group;" ::: "memory");  // one group per box, even past N
        }
      } else if (r < rows) {
#pragma unroll
        for (int k = 0; k < 8; ++k)
          if (col + 8 * k < N)
            *reinterpret_cast<uint4*>(orow + col + 8 * k) = make_uint4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
      }
    }
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  cluster_sync_all();  // neither CTA frees its tensor memory or retires while the pair still uses them
  if (warp == kProducerWarps) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(TMEM_COLS) : "memory");
  }
}

template <int MODE, bool DENSE>
cudaError_t launch_w4a16(const DevInfo& d, const uint16_t* x, const int32_t* lhs, const int32_t* rhs, int64_t R,
                         const uint32_t* w, const void* scales, const uint16_t* biases, const float* gs_w, int64_t E,
                         int64_t N, int64_t K, int group, uint16_t* out, int inject, cudaStream_t s) {
  using C = Cfg<MODE, DENSE>;
  if (C::kSmemBytes > d.smem_optin) return cudaErrorInvalidValue;
  auto fn = encode_fn();
  if (!fn) return cudaErrorInvalidValue;
  auto map2d = [&](CUtensorMap* m, const void* p, int64_t inner, int64_t outer, uint32_t bi, uint32_t bo,
                   CUtensorMapSwizzle sw) {
    cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
    cuuint64_t strides[1] = {(cuuint64_t)inner * 2};
    cuuint32_t box[2] = {bi, bo};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  };
  CUtensorMap tmX, tmO;
  // activations [rows, K]: boxes of 256 (qmm) or 128 (gather_qmm) rows x 64 elements
  // (128 bytes), 128-byte swizzle (gather_qmm: x's row count is not an argument --
  // the map is open-ended and only boxes of rows the routing names are loaded);
  // output [R, N]: TMA stores of 32 rows x 64 columns, 128-byte swizzle
  if (!map2d(&tmX, x, K, DENSE ? R : (int64_t)1 << 30, BK, DENSE ? TM : BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !map2d(&tmO, out, N, R, 64, 32, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(w4a16_kernel<MODE, DENSE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)C::kSmemBytes);
  if (e != cudaSuccess) return e;
  // gather: an upper bound on the per-expert tiles; slots past the last tile exit at once
  const int64_t m_tiles = DENSE ? (R + TM - 1) / TM : (R + TM - 1) / TM + E;
  dim3 grid((unsigned)((N + BN - 1) / BN), (unsigned)m_tiles);
  w4a16_kernel<MODE, DENSE><<<grid, kThreads, C::kSmemBytes, s>>>(tmX, tmO, x, lhs, rhs, (int)R, w, scales,
                                                                   biases, gs_w, (int)E, (int)N, (int)K, group, out,
                                                                   d.err, inject);
  return cudaGetLastError();
}

// Clusters of two qmm_pair_kernel<MODE> CTAs that can be resident at once (0:
// the pair kernel cannot run here and qmm takes the one-SM kernel).
template <int MODE>
int qmm_pair_clusters(const DevInfo& d) {
  static std::mutex mu;
  static int cache[64];
  static bool have[64];
  if (d.device < 0 || d.device >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (have[d.device]) return cache[d.device];
  int n = 0;
  const int smem = (int)PairQ<MODE>::kSmemBytes;
  if (smem <= d.smem_optin &&
      cudaFuncSetAttribute(qmm_pair_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) == cudaSuccess) {
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
    if (cudaOccupancyMaxActiveClusters(&n, qmm_pair_kernel<MODE>, &cfg) != cudaSuccess) {
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
cudaError_t launch_qmm_pair(const DevInfo& d, const uint16_t* x, int64_t M, const uint32_t* w, const void* scales,
                            const uint16_t* biases, const float* gs_w, int64_t N, int64_t K, int group,
                            uint16_t* out, int inject, cudaStream_t s) {
  using P = PairQ<MODE>;
  auto fn = encode_fn();
  if (!fn) return cudaErrorInvalidValue;
  auto map2d = [&](CUtensorMap* m, const void* p, int64_t inner, int64_t outer, uint32_t bi, uint32_t bo) {
    cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
    cuuint64_t strides[1] = {(cuuint64_t)inner * 2};
    cuuint32_t box[2] = {bi, bo};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  };
  CUtensorMap tmX, tmO;
  // activations [M, K]: boxes of 128 rows x 64 elements; output [M, N]: stores of 32 rows x 64 columns
  if (!map2d(&tmX, x, K, M, BK, BM) || !map2d(&tmO, out, N, M, 64, 32)) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * ((N + BN - 1) / BN)), (unsigned)((M + kPairRows - 1) / kPairRows));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = P::kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, qmm_pair_kernel<MODE>, tmX, tmO, (int)M, w, scales, biases, gs_w, (int)N, (int)K,
                            group, out, d.err, inject);
}

// out[i, :] = x[idx[i], :]: one warp per row at a time, 16-byte pieces; an index
// outside [0, x_rows) leaves its row unwritten and is reported.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* __restrict__ x, int64_t x_rows,
                                                          const int32_t* __restrict__ idx, int64_t R, int pieces,
                                                          uint4* __restrict__ out, unsigned* __restrict__ err) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t i = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); i < R; i += warps) {
    const int64_t src = __ldg(idx + i);
    if (src < 0 || src >= x_rows) {
      if (lane == 0) record_error(err, kErrIndex);
      continue;
    }
    const uint4* a = x + src * pieces;
    uint4* o = out + i * pieces;
    int c = lane;
    for (; c + 96 < pieces; c += 128) {  // four 16-byte loads in flight per lane
      const uint4 v0 = ld_stream_v4(a + c), v1 = ld_stream_v4(a + c + 32), v2 = ld_stream_v4(a + c + 64),
                  v3 = ld_stream_v4(a + c + 96);
      o[c] = v0;
      o[c + 32] = v1;
      o[c + 64] = v2;
      o[c + 96] = v3;
    }
    for (; c < pieces; c += 32) o[c] = ld_stream_v4(a + c);
  }
}

}  // namespace

cudaError_t launch_gather_rows(const DevInfo& d, const uint16_t* x, int64_t x_rows, const int32_t* idx, int64_t R,
                               int64_t K, uint16_t* out, cudaStream_t s) {
  const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>((R + 7) / 8, (int64_t)d.sm_count * 8));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gather_rows_kernel, reinterpret_cast<const uint4*>(x), x_rows, idx, R, (int)(K / 8),
                            reinterpret_cast<uint4*>(out), d.err);
}

cudaError_t launch_gather_qmm(const DevInfo& d, const uint16_t* x, const int32_t* lhs, const int32_t* rhs, int64_t R,
                              const uint32_t* w, const void* scales, const uint16_t* biases, const float* gs_w,
                              int64_t E, int64_t N, int64_t K, int mode, int group, uint16_t* out, int inject_timeout,
                              cudaStream_t s) {
  if (mode == 1)
    return launch_w4a16<1, false>(d, x, lhs, rhs, R, w, scales, biases, gs_w, E, N, K, group, out, inject_timeout, s);
  if (mode == 2)
    return launch_w4a16<2, false>(d, x, lhs, rhs, R, w, scales, biases, gs_w, E, N, K, group, out, inject_timeout, s);
  return launch_w4a16<0, false>(d, x, lhs, rhs, R, w, scales, biases, gs_w, E, N, K, group, out, inject_timeout, s);
}

cudaError_t launch_qmm(const DevInfo& d, const uint16_t* x, int64_t M, const uint32_t* w, const void* scales,
                       const uint16_t* biases, const float* gs_w, int64_t N, int64_t K, int mode, int group,
                       uint16_t* out, int inject_timeout, cudaStream_t s) {
  // CTA pairs wherever a pair can be resident (512 x 256 tiles, each SM
  // dequantizing 128 weight rows); the one-SM kernel otherwise
  if (mode == 1 && qmm_pair_clusters<1>(d) > 0)
    return launch_qmm_pair<1>(d, x, M, w, scales, biases, gs_w, N, K, group, out, inject_timeout, s);
  if (mode == 2 && qmm_pair_clusters<2>(d) > 0)
    return launch_qmm_pair<2>(d, x, M, w, scales, biases, gs_w, N, K, group, out, inject_timeout, s);
  if (mode == 0 && qmm_pair_clusters<0>(d) > 0)
    return launch_qmm_pair<0>(d, x, M, w, scales, biases, gs_w, N, K, group, out, inject_timeout, s);
  if (mode == 1)
    return launch_w4a16<1, true>(d, x, nullptr, nullptr, M, w, scales, biases, gs_w, 1, N, K, group, out,
                                 inject_timeout, s);
  if (mode == 2)
    return launch_w4a16<2, true>(d, x, nullptr, nullptr, M, w, scales, biases, gs_w, 1, N, K, group, out,
                                 inject_timeout, s);
  return launch_w4a16<0, true>(d, x, nullptr, nullptr, M, w, scales, biases, gs_w, 1, N, K, group, out,
                               inject_timeout, s);
}

}  // namespace fp4
