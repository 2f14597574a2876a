// common.cuh -- shared device helpers for libfp4gb300 (sm_103a only).
//
// Everything here is written for the GB300 tensor-memory/TMA execution model:
// mbarrier waits are bounded (a wait that gives up records an error word and
// returns false; no trap, no endless loop), conversions use the hardware
// e2m1x2 / e4m3x2 converters, and fp32 steps that must match the quantization
// rule bit for bit use the explicitly rounded intrinsics (__fmul_rn, __fdiv_rn,
// __frcp_rn) so the compiler cannot contract or approximate them.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ != 1030 || !defined(__CUDA_ARCH_FEAT_SM103_ALL))
#error "libfp4gb300 is built for sm_103a only (-gencode arch=compute_103a,code=sm_103a)"
#endif

namespace fp4 {

// Error word bits: a bounded wait expired; a kernel found an index argument
// outside its contract (gather_qmm's expert ids).
constexpr unsigned kErrTimeout = 1u;
constexpr unsigned kErrIndex = 2u;

// Limit of one bounded wait, in SM clock cycles (~0.5 s at 2 GHz).  A thread
// whose wait expired once stops waiting (later waits try once and return), so
// a broken pipeline costs one limit per thread, not one per stage.
constexpr long long kWaitLimitCycles = 1000000000LL;

__device__ __forceinline__ void record_error(unsigned* err, unsigned code) {
  if (err) atomicOr(err, code);
}

// ---------------------------------------------------------------- bf16 ----
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Round an fp32 value to the nearest-even bf16 (returns the 16 bits).
__device__ __forceinline__ uint32_t f32_to_bf16_rn(float v) {
  uint16_t r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(v));
  return r;
}

__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// --------------------------------------------------------- 4-bit codecs ----
// Two fp32 values -> one byte of two e2m1 codes: `lo` in bits 0..3, `hi` in
// bits 4..7 (round to nearest even, saturate to +-6, sign kept).
__device__ __forceinline__ uint32_t e2m1x2_rn(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 b;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b, %1, %2;\n\t"
      "cvt.u32.u8 %0, b;\n\t}"
      : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Eight fp32 values -> eight e2m1 codes (round to nearest even, saturating),
// code k in bits 4k .. 4k + 3: four converts whose bytes are packed by moves.
__device__ __forceinline__ uint32_t e2m1x8_rn(const float (&v)[8]) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t.reg .b16 h0, h1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b16 h0, {b0, b1};\n\t"
      "mov.b16 h1, {b2, b3};\n\t"
      "mov.b32 %0, {h0, h1};\n\t}"
      : "=r"(r)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return r;
}

// One byte of two e2m1 codes -> f16x2 (low code in the low half).
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t r;
  asm("{\n\t.reg .b8 b;\n\t"
      "cvt.u8.u32 b, %1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b;\n\t}"
      : "=r"(r) : "r"(byte));
  return r;
}

__device__ __forceinline__ float f16_lo_to_f32(uint32_t h2) {
  float f;
  asm("{\n\t.reg .f16 l, h;\n\tmov.b32 {l, h}, %1;\n\tcvt.f32.f16 %0, l;\n\t}" : "=f"(f) : "r"(h2));
  return f;
}
__device__ __forceinline__ float f16_hi_to_f32(uint32_t h2) {
  float f;
  asm("{\n\t.reg .f16 l, h;\n\tmov.b32 {l, h}, %1;\n\tcvt.f32.f16 %0, h;\n\t}" : "=f"(f) : "r"(h2));
  return f;
}

// fp32 -> E4M3 byte (round to nearest even, saturate to 448).
__device__ __forceinline__ uint32_t e4m3_rn(float v) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
  return r & 0xFFu;
}

// E4M3 byte -> fp32 (exact, through the hardware e4m3x2 -> f16x2 converter).
__device__ __forceinline__ float e4m3_to_f32(uint32_t byte) {
  uint32_t h2;
  uint16_t b = (uint16_t)(byte & 0xFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(b));
  return f16_lo_to_f32(h2);
}

// 2^e as fp32 for e in [-127, 127] (2^-127 is a subnormal).
__device__ __forceinline__ float exp2i_f32(int e) {
  return e >= -126 ? __uint_as_float((uint32_t)(e + 127) << 23) : __uint_as_float(0x00400000u);
}

// E8M0 byte -> fp32 (0xFF, NaN, is outside the contract).
__device__ __forceinline__ float e8m0_to_f32(uint32_t byte) { return exp2i_f32((int)(byte & 0xFFu) - 127); }

// ------------------------------------------------- block quantization rule ----
// The fp_quantize rule for one block from the bits of its largest |x| (bf16
// magnitude bits, mb): the multiplier that maps x to e2m1 (q = e2m1_rn_sat(x *
// mul)), the scale byte stored, and the scale's value.
//   NVFP4 (MODE 2, E4M3 per 16): b = max|x|, s8 = E4M3_rn_sat(b / fl(6 gs)) (0 when
//     b = 0), mul = 1 / fl(s8 gs) (0 when that product is 0).
//   MXFP4 (MODE 1, E8M0 per 32): se = clamp(floor(log2 b) - 2, -127, 127) (-127 when
//     b = 0), byte = se + 127, mul = 2^-se.
//
// The NVFP4 division b / fl(6 gs) has one divisor per tensor, so its
// correctly rounded reciprocal r = 1/p is formed once (Nvfp4Div) and each block
// divides by Markstein's correction: q0 = fl(b r), e = b - q0 p (exact by
// FMA), q = fl(q0 + e r), which is fl(b / p) when p, 1/p and b are normal
// enough that e does not underflow (b >= 2^-100) and q0 lies in [2^-64, 1024).
// Outside that range q0 itself is returned: the block scale is only its e4m3
// rounding, which saturates at 448 above 1024 and is 0 below 2^-10.  Checked
// exhaustively on the CPU against correctly rounded division for every pair of
// bf16 amax (gs = fl(amax / 2688)) and bf16 block maximum b <= amax, and for
// every bf16 b against 20,000 random normal divisors (a quarter of them with an
// all-ones mantissa): every e4m3 result agrees.
struct Nvfp4Div {
  float p, r;
  bool fast;
};

__device__ __forceinline__ Nvfp4Div nvfp4_div(float gs) {
  Nvfp4Div d;
  d.p = __fmul_rn(6.0f, gs);
  d.r = __frcp_rn(d.p);
  d.fast = d.p >= 0x1p-126f && d.p < 0x1p126f;  // p and 1/p normal
  return d;
}

__device__ __forceinline__ float nvfp4_block_div(float b, const Nvfp4Div& d) {
  if (!d.fast || b < 0x1p-100f) return __fdiv_rn(b, d.p);
  const float q0 = __fmul_rn(b, d.r);
  if (!(q0 < 1024.0f) || q0 < 0x1p-64f) return q0;
  return __fmaf_rn(__fmaf_rn(-q0, d.p, b), d.r, q0);
}

// Two round-to-nearest fp32 products in one packed instruction (each lane is
// an IEEE multiply, the same as __fmul_rn).
__device__ __forceinline__ void fmul2_rn(float a0, float a1, float m, float& r0, float& r1) {
  asm("{\n\t.reg .b64 a, b, d;\n\t"
      "mov.b64 a, {%2, %3};\n\t"
      "mov.b64 b, {%4, %4};\n\t"
      "mul.rn.f32x2 d, a, b;\n\t"
      "mov.b64 {%0, %1}, d;\n\t}"
      : "=f"(r0), "=f"(r1) : "f"(a0), "f"(a1), "f"(m));
}

template <int MODE>
__device__ __forceinline__ void block_scale_rule(uint32_t mb, float gs, const Nvfp4Div& dv, float& mul,
                                                 uint32_t& sbyte, float& sval) {
  if (MODE == 2) {
    const float b = __uint_as_float(mb << 16);
    const float sc = (b == 0.0f) ? 0.0f : nvfp4_block_div(b, dv);
    sbyte = e4m3_rn(sc);
    sval = e4m3_to_f32(sbyte);
    const float dd = __fmul_rn(sval, gs);
    mul = (dd == 0.0f) ? 0.0f : __frcp_rn(dd);
  } else {
    int se = -127;
    if (mb != 0) {
      const int E = (int)(mb >> 7);
      const int e = (E == 0) ? (-133 + (31 - __clz((int)(mb & 0x7Fu)))) : (E - 127);
      se = min(max(e - 2, -127), 127);
    }
    sbyte = (uint32_t)(se + 127);
    mul = exp2i_f32(-se);
    sval = exp2i_f32(se);
  }
}

template <int MODE>
__device__ __forceinline__ void block_scale_rule(uint32_t mb, float gs, float& mul, uint32_t& sbyte,
                                                 float& sval) {
  block_scale_rule<MODE>(mb, gs, nvfp4_div(gs), mul, sbyte, sval);
}

// Largest bf16 magnitude (bits) of the eight values of a 16-byte piece.
__device__ __forceinline__ uint32_t max_mag8(uint4 v) {
  uint32_t m2 = __vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu);
  m2 = __vmaxu2(m2, v.z & 0x7FFF7FFFu);
  m2 = __vmaxu2(m2, v.w & 0x7FFF7FFFu);
  return max(m2 & 0xFFFFu, m2 >> 16);
}

// fp_quantize then fp_dequantize of eight bf16 values of one block: each
// value becomes bf16_rn(fl(fl(e2m1(q) * sval) * gs)) with q = e2m1_rn_sat(x * mul)
// (gs = 1 for MXFP4 or without a global scale; the multiply by 1 is exact).
__device__ __forceinline__ uint4 quant_dequant8(uint4 v, float mul, float sval, float gs) {
  const uint32_t in[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t code2 = e2m1x2_rn(__fmul_rn(bf16_lo(in[j]), mul), __fmul_rn(bf16_hi(in[j]), mul));
    const uint32_t h2 = e2m1x2_to_f16x2(code2);
    o[j] = pack_bf16x2_rn(__fmul_rn(__fmul_rn(f16_lo_to_f32(h2), sval), gs),
                          __fmul_rn(__fmul_rn(f16_hi_to_f32(h2), sval), gs));
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// ---------------------------------------------------------- tiled scales ----
__device__ __forceinline__ int64_t tiled_scale_offset(int64_t r, int64_t c, int64_t padded_cols) {
  int64_t tile = (r >> 7) * (padded_cols >> 2) + (c >> 2);
  int64_t rr = r & 127;
  return (tile << 9) + ((rr & 31) << 4) + ((rr >> 5) << 2) + (c & 3);
}

// ------------------------------------------------------------ memory ops ----
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// -------------------------------------------------------------- mbarrier ----
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}"
               :: "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}"
               :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar_addr, uint32_t parity) {
  uint32_t ok;
  asm volatile("{\n\t.reg .pred p;\n\t"
               "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
               "selp.u32 %0, 1, 0, p;\n\t}"
               : "=r"(ok) : "r"(bar_addr), "r"(parity) : "memory");
  return ok != 0;
}

// Bounded wait for phase `parity` of `bar`.  Returns false (records
// kErrTimeout, sets `failed`) if the phase did not complete within `limit`
// cycles; once `failed` is set, later calls only test the phase once.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned* err, bool& failed,
                                          long long limit = kWaitLimitCycles) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  if (failed) return false;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(a, parity)) return true;
    if (clock64() - t0 > limit) {
      record_error(err, kErrTimeout);
      failed = true;
      return false;
    }
  }
}

// --------------------------------------------------------------- TMA -------
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const void* tmap, uint64_t* bar, int x,
                                            int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];"
      :: "r"(smem_u32(smem_dst)), "l"(tmap), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* smem_dst, const void* tmap, uint64_t* bar, int x, int y,
                                            int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];"
      :: "r"(smem_u32(smem_dst)), "l"(tmap), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// Untiled bulk copy global -> shared (16-byte aligned addresses, size % 16 == 0).
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      :: "r"(smem_u32(smem_dst)), "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" :: "l"(tmap) : "memory");
}

__device__ __forceinline__ uint32_t elect_one_sync() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .b32 r;\n\t.reg .pred p;\n\t"
      "elect.sync r|p, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred;
}

}  // namespace fp4
