/*
 * fp4_oracle.h -- plain, slow CPU oracle for block-scaled 4-bit quantization
 * (NVFP4, MXFP4, affine-4) and the matmuls built on it.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this library: it is used by tests/, by __graft_entry__.smoke() and by the
 * cpu_baseline leg of bench.py.  It shares no source, header, table or helper
 * with the CUDA library in block_scaled_fp4_fp_gb300/csrc.
 *
 * Conventions (all stated independently of the CUDA side):
 *   - bf16 values are passed as raw 16-bit patterns (uint16_t).
 *   - A 4-bit code is e2m1: bit 3 sign, bits 2..1 exponent (bias 1), bit 0
 *     mantissa.  Element k of a row lives in 32-bit word k/8, nibble k%8, the
 *     low nibble first.
 *   - mode: 0 = affine, 1 = MXFP4 (group 32, E8M0 scale), 2 = NVFP4 (group 16,
 *     E4M3 scale, optional fp32 global scale in multiplier form amax/2688).
 *   - Linear scales are row-major [rows, cols/group].  The tiled layout is the
 *     128x4 tile layout described with orc_tiled_offset().
 *   - Every fp32 step is one IEEE round-to-nearest-even operation (the file is
 *     compiled with -ffp-contract=off).  Matmuls accumulate in fp64.
 *
 * Parity status of each function is given in its comment ("pinned by ...").
 */
#ifndef FP4_ORACLE_H
#define FP4_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- scalar codecs ---------------------------------------------------- */
double   orc_e2m1_decode(unsigned code);
unsigned orc_e2m1_encode(float v);
double   orc_e4m3_decode(unsigned byte);
unsigned orc_e4m3_encode(float v);
double   orc_e8m0_decode(unsigned byte);
double   orc_bf16_to_double(uint16_t b);
uint16_t orc_bf16_from_double(double v);
uint16_t orc_bf16_from_float(float v);

/* ---- per-tensor global scale and alpha -------------------------------- */
float orc_amax(const uint16_t* x, int64_t n);
float orc_global_scale(const uint16_t* x, int64_t n);        /* fl(amax / 2688) */
float orc_alpha_from_amax(float amax_x, float amax_w);         /* amax_x*amax_w/(448*6)^2 */

/* ---- quantizers (linear scales) --------------------------------------- */
void orc_nvfp4_quantize(const uint16_t* x, int64_t rows, int64_t cols,
                        const float* global_scale, uint32_t* q, uint8_t* scales);
void orc_mxfp4_quantize(const uint16_t* x, int64_t rows, int64_t cols,
                        uint32_t* q, uint8_t* scales);
void orc_affine_quantize(const uint16_t* w, int64_t rows, int64_t cols, int group,
                         uint32_t* q, uint16_t* scales, uint16_t* biases);

/* ---- stochastic-rounding quantizers (see fp4_oracle.c for the contract) -- */
void     orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);
uint32_t orc_sr_word(uint64_t seed, uint64_t offset, uint64_t e);
unsigned orc_e2m1_encode_sr(float v, uint32_t u);
void orc_nvfp4_quantize_sr(const uint16_t* x, int64_t rows, int64_t cols, const float* global_scale,
                           uint64_t seed, uint64_t offset, uint32_t* q, uint8_t* scales);
void orc_mxfp4_quantize_sr(const uint16_t* x, int64_t rows, int64_t cols, uint64_t seed, uint64_t offset,
                           uint32_t* q, uint8_t* scales);

/* ---- scale tile layout ------------------------------------------------ */
int64_t orc_padded_rows(int64_t rows);
int64_t orc_padded_cols(int64_t cols);
int64_t orc_tiled_offset(int64_t r, int64_t c, int64_t padded_cols);
void orc_tile_scales(const uint8_t* linear, int64_t rows, int64_t cols, uint8_t* tiled);
void orc_untile_scales(const uint8_t* tiled, int64_t rows, int64_t cols, uint8_t* linear);

/* ---- dequantize --------------------------------------------------------- */
/* Exact value of every element in fp64 (no rounding). */
void orc_dequantize_f64(const uint32_t* q, const void* scales, const uint16_t* biases,
                        int64_t rows, int64_t cols, int mode, int group,
                        const float* global_scale, double* out);
/* The fp32 value fl(code*scale*gs) (affine: fl(q*s + b)) rounded RNE to bf16. */
void orc_dequantize_bf16(const uint32_t* q, const void* scales, const uint16_t* biases,
                         int64_t rows, int64_t cols, int mode, int group,
                         const float* global_scale, uint16_t* out);

/* ---- matmuls (fp64 accumulation) -------------------------------------- */
/* y[i] = sum_k x[k] * deq(W)[rows[i], k]; rows == NULL means all N rows. */
void orc_qmv(const uint16_t* x, const uint32_t* w, const void* scales, const uint16_t* biases,
             const float* global_scale_w, int64_t N, int64_t K, int mode, int group,
             const int64_t* rows, int64_t nrows, double* y);
/* out[i,j] = alpha * sum_k c(xq)[mi,k]*sx * c(wq)[nj,k]*sw over the listed rows
 * mi of xq and rows nj of wq (NULL lists mean all); linear scales; mode 1 or 2. */
void orc_qqmm(const uint32_t* xq, const uint8_t* sx, const uint32_t* wq, const uint8_t* sw,
              float alpha, int64_t M, int64_t N, int64_t K, int mode,
              const int64_t* mrows, int64_t nm, const int64_t* ncols, int64_t nn, double* out);
/* out[i, n] = sum_k x[m_i, k] * deq(W)[n, k] (with the NVFP4 weight global scale) over
 * the listed rows m_i of x [M, K] (NULL means all), every column n. */
void orc_qmm(const uint16_t* x, int64_t M, const uint32_t* w, const void* scales, const uint16_t* biases,
             const float* global_scale_w, int64_t N, int64_t K, int mode, int group,
             const int64_t* rows, int64_t nrows, double* out);
/* out[i, n] = sum_k x[lhs[r_i], k] * deq(W[rhs[r_i]])[n, k] for the listed routed
 * rows r_i (NULL means all R), all N columns.  W is [E, N, K] packed. */
void orc_gather_qmm(const uint16_t* x, const int32_t* lhs, const int32_t* rhs, int64_t R,
                    const uint32_t* w, const void* scales, const uint16_t* biases,
                    int64_t E, int64_t N, int64_t K, int mode, int group,
                    const int64_t* rows, int64_t nrows, double* out);

int orc_num_threads(void);

#ifdef __cplusplus
}
#endif
#endif
