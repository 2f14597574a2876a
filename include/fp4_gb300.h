/*
 * fp4_gb300.h -- C ABI of libfp4gb300: block-scaled 4-bit quantization and
 * quantized matmul on one NVIDIA GB300 (sm_103a).
 *
 * Sources (pages cited by title and section):
 *   [P1] "perf(cuda): enable hardware NVFP4/MXFP4 conversion on Blackwell
 *        builds" -- fp_quantize: MXFP4 and NVFP4 share one template; e2m1 by
 *        cvt.rn.satfinite.e2m1x2.f32 on sm_100a-class targets.
 *   [P2] "epic: NVIDIA Volta (sm_70) inference acceleration program #1536" --
 *        Baseline and Diagnosis 3: qmv over affine 4-bit group-64 weights, the
 *        decode-step weight stream; Diagnosis 1 and 5: gather_gemm / grouped
 *        GEMM for MoE.
 *   [P3] "mlx 0.30.7.3 -> 0.30.7.6" -- qqmm.cpp (QQMatmul::eval_gpu,
 *        quantize_input: packed codes [.., K*bits/32] uint32, scales uint8,
 *        W always transposed [N, K]), qqmm_utils.h (128x4 scale tiles, zero
 *        padding, 16-byte aligned start), qqmm_utils.cu (alpha =
 *        amax_x*amax_w/(448*6)^2, beta = 0), quantized.cpp
 *        (fast::Quantize::eval_gpu: optional NVFP4 global scale).
 *   [P4] "mlx: opt-in dense GEMM for nvfp4 prefill ... - #287" -- global scale
 *        representations (multiplier m versus m*2688).
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     keeps none of them after the call returns and allocates nothing.
 *   - bf16 tensors are raw bfloat16 bit patterns (fp4_bf16), row-major and
 *     contiguous.  Packed 4-bit codes are uint32 words: element k of a row is
 *     word k/8, nibble k%8, low nibble first (8 codes per word).
 *   - Work is enqueued on `stream` (stream-ordered, asynchronous).  Arguments
 *     are validated on the host before anything is launched; an invalid call
 *     launches nothing and returns a non-OK status.  No C++ exception crosses
 *     the ABI.  Launch failures return FP4_ERR_CUDA.  A device-side wait that
 *     gives up (bounded spin) records FP4_ERR_TIMEOUT, which
 *     fp4_check_device_error() reports.
 *   - Every size (n, rows, cols, N, K, M, R, E) must be at least 1: an empty
 *     problem returns FP4_ERR_INVALID_ARG and launches nothing.
 *   - NVFP4: e2m1 codes, groups of 16, E4M3 block scales, optional fp32 global
 *     scale gs in the multiplier form gs = amax/2688 (2688 = 448*6).
 *     MXFP4: e2m1 codes, groups of 32, E8M0 block scales.
 *     Affine: unsigned 4-bit q, groups of 32/64/128, bf16 scale and bias,
 *     w = q*scale + bias.
 */
#ifndef FP4_GB300_H
#define FP4_GB300_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t fp4_bf16; /* raw bfloat16 bits */

typedef enum {
  FP4_OK = 0,
  FP4_ERR_INVALID_ARG = 1,  /* null pointer, negative or inconsistent size */
  FP4_ERR_UNSUPPORTED = 2,  /* mode/bits/group combination or device not supported */
  FP4_ERR_ALIGNMENT = 3,    /* a pointer or a row pitch breaks the alignment rule */
  FP4_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
  FP4_ERR_TIMEOUT = 5       /* a bounded device wait expired (see fp4_check_device_error) */
} fp4_status;

typedef enum { FP4_MODE_AFFINE = 0, FP4_MODE_MXFP4 = 1, FP4_MODE_NVFP4 = 2 } fp4_mode;

/* Scale layouts.  LINEAR: row-major [rows, cols/group].
 * TILED_128x4 [P3 qqmm_utils.h]: rows padded to a multiple of 128 and scale
 * columns to a multiple of 4; byte (r, c) sits at
 *   ((r/128)*(Cp/4) + c/4)*512 + (r%32)*16 + ((r%128)/32)*4 + c%4
 * (Cp = padded scale columns), every padding byte is zero, total Rp*Cp bytes. */
typedef enum { FP4_SCALES_LINEAR = 0, FP4_SCALES_TILED_128x4 = 1 } fp4_scale_layout;

/* Checks that `device` is compute capability 10.3 (GB300) and caches its
 * properties.  Every other entry point initializes the current device lazily,
 * so calling this is optional; it is the place to learn FP4_ERR_UNSUPPORTED. */
fp4_status fp4_init(int device);

/* Static string for a status code; never NULL. */
const char* fp4_status_string(fp4_status status);

/* Synchronizes `stream`, then reports and clears the device error word of the
 * current device: FP4_ERR_TIMEOUT if any bounded wait of an earlier launch
 * expired since the last check, FP4_ERR_INVALID_ARG if a kernel found an index
 * argument outside its contract (gather_qmm's expert ids), FP4_ERR_CUDA if the
 * stream reports an error, else FP4_OK. */
fp4_status fp4_check_device_error(cudaStream_t stream);

/* Padded scale-tile dimensions for `rows` x `scale_cols` scales
 * [P3 qqmm_utils.h get_padded_scale_dims]: rows up to a multiple of 128,
 * columns up to a multiple of 4. */
void fp4_padded_scale_dims(int64_t rows, int64_t scale_cols, int64_t* padded_rows,
                           int64_t* padded_cols);

/* Bytes of device workspace fp4_amax_global_scale needs for n elements. */
size_t fp4_amax_workspace_bytes(int64_t n);

/* a1: tensor amax and NVFP4 global scale [P3 quantize_input / compute_qqmm_pointers,
 * P4 global-scale representation].
 *   x        bf16[n], 16-byte aligned, n >= 1
 *   gs_out   device fp32 scalar: fl(amax/2688), the multiplier form m
 *   amax_out device fp32 scalar or NULL: max |x| (MLX's m*2688 form)
 *   ws       device scratch of ws_bytes >= fp4_amax_workspace_bytes(n) bytes;
 *            no initial contents needed; not read after the call completes.
 * NaN inputs give an unspecified result. */
fp4_status fp4_amax_global_scale(const fp4_bf16* x, int64_t n, float* gs_out, float* amax_out,
                                 void* ws, size_t ws_bytes, cudaStream_t stream);

/* a2-a4: fp_quantize [P1; P3 qqmm.cpp quantize_input, quantized.cpp].
 *   x            bf16[rows, cols], 16-byte aligned
 *   mode, bits, group_size: (NVFP4, 4, 16) or (MXFP4, 4, 32); affine quantize is
 *                not provided (FP4_ERR_UNSUPPORTED)
 *   global_scale device fp32 scalar gs (NVFP4 only) or NULL (gs = 1)
 *   xq           uint32[rows, cols/8] packed codes, 8-byte (NVFP4) / 16-byte (MXFP4) aligned
 *   scales       uint8 E4M3/E8M0 block scales in `layout`; for TILED_128x4 the
 *                whole padded buffer (Rp*Cp bytes) is written, padding with 0
 * Per NVFP4 group: b = max|x|, s8 = E4M3_rn_sat(b/(6*gs)) (0 when b = 0),
 *   q = e2m1_rn_sat(x * (1/(s8*gs))) (0 codes with their sign when s8*gs = 0).
 * Per MXFP4 group: se = clamp(floor(log2 b) - 2, -127, 127) (-127 when b = 0),
 *   byte = se + 127, q = e2m1_rn_sat(x * 2^-se).
 * Requires cols % group_size == 0 and rows >= 1. */
fp4_status fp4_quantize(const fp4_bf16* x, int64_t rows, int64_t cols, fp4_mode mode, int bits,
                        int group_size, const float* global_scale, uint32_t* xq, uint8_t* scales,
                        fp4_scale_layout layout, cudaStream_t stream);

/* fp_quantize with stochastic rounding [P1: the NVFP4/MXFP4 quantizer's USE_SR
 * template parameter, which needs the Blackwell converters; the pages state
 * neither the rule nor the random numbers, so both are fixed here].
 * Arguments as fp4_quantize, plus seed and offset.  Block scales are exactly
 * fp4_quantize's.  Each element v = x * mul (mul as fp4_quantize) is rounded to
 * one of its two e2m1 neighbours lo <= |v| < hi: up when the top 24 bits of its
 * random word are below floor(2^24 (|v| - lo) / (hi - lo)), so the expected
 * value is v (to 2^-24 of the step); |v| >= 6 gives 6 and the sign is kept.
 * The random word of element e = r * cols + c is word e % 4 of Philox4x32-10
 * (Salmon et al., "Parallel random numbers: as easy as 1, 2, 3", SC 2011) at
 * the 128-bit counter offset + floor(e / 4) (32-bit words little-endian) under
 * the key (low 32 bits of seed, high 32 bits): independent of the launch
 * configuration, so a call is reproducible, and successive calls that advance
 * offset by ceil(rows * cols / 4) never reuse a word. */
fp4_status fp4_quantize_sr(const fp4_bf16* x, int64_t rows, int64_t cols, fp4_mode mode, int bits,
                           int group_size, const float* global_scale, uint64_t seed, uint64_t offset, uint32_t* xq,
                           uint8_t* scales, fp4_scale_layout layout, cudaStream_t stream);

/* a5: fp_dequantize / affine_dequantize [P3 quantized.cpp].
 *   wq      uint32[rows, cols/8]
 *   scales  NVFP4/MXFP4: uint8 block scales in `layout`; affine: bf16[rows, cols/group]
 *           (linear layout only)
 *   biases  affine: bf16[rows, cols/group]; must be NULL otherwise
 *   global_scale NVFP4 only, device fp32 or NULL
 *   out     bf16[rows, cols], 16-byte aligned
 * Each element is the fp32 value code*scale*gs (affine q*scale + bias) rounded
 * to nearest-even bf16. */
fp4_status fp4_dequantize(const uint32_t* wq, const void* scales, const fp4_bf16* biases,
                          int64_t rows, int64_t cols, fp4_mode mode, int bits, int group_size,
                          const float* global_scale, fp4_scale_layout layout, fp4_bf16* out,
                          cudaStream_t stream);

/* a6: qmv, the M = 1 decode GEMV [P2 Baseline, Diagnosis 3; P3 qqmm.cpp fp_qmv route].
 *   y[n] = sum_k x[k] * deq(W)[n, k]   (fp32 accumulation, bf16 output)
 *   x       bf16[K], 16-byte aligned
 *   w       uint32[N, K/8] (W stored [N, K]), 16-byte aligned
 *   scales  linear block scales: uint8[N, K/group] (NVFP4/MXFP4) or bf16 (affine)
 *   biases  affine: bf16[N, K/group]; NULL otherwise
 *   global_scale_w NVFP4 only: device fp32 gs of W, multiplied in the epilogue, or NULL
 *   y       bf16[N]
 * Requires K % 32 == 0 and K % group_size == 0.
 * Launch order: qmv uses programmatic dependent launch and may read w and its
 * scales before the kernel launched just before it on the stream has finished;
 * x, global_scale_w and y are touched only after that kernel completes.  No
 * kernel of this library writes weights and releases its dependents early, so
 * any sequence of calls through this header is ordered; a caller's own kernel
 * that writes w and triggers its dependents early must not directly precede qmv.
 * A NaN or infinity in x gives non-finite rows (tensor-core path, NVFP4 and MXFP4: NaN). */
fp4_status qmv(const fp4_bf16* x, const uint32_t* w, const void* scales, const fp4_bf16* biases,
               const float* global_scale_w, int64_t N, int64_t K, fp4_mode mode, int bits,
               int group_size, fp4_bf16* y, cudaStream_t stream);

/* The weights of one GEMV launch: up to 4 matrices of the same K, each given as
 * qmv takes it (biases: affine only; global_scale_w: NVFP4 only, may be NULL). */
typedef struct fp4_matrix_group {
  int count; /* 1 .. 4 */
  const uint32_t* w[4];
  const void* scales[4];
  const fp4_bf16* biases[4];
  const float* global_scale_w[4];
  int64_t N[4];
  int64_t K;
} fp4_matrix_group;

/* qmv_grouped: the decode GEMV of one x against the matrices of `mats` in one
 * launch -- the projections that multiply the same activation (q, k and v;
 * gate and up) stored as separate matrices [P2 Baseline: the decode step is the
 * qmv weight stream; grouping them pays the per-launch fixed cost once].
 *   y[i] = x . deq(W_i)^T  for i < mats->count (each y[i] as qmv computes it);
 *   y: a HOST array of mats->count device pointers.
 * prefetch_next (NULL: none): the weights of the GEMV the caller launches next
 * on this stream, same mode.  A hint: once this launch has issued its own
 * weight loads, it warms L2 with the first stages that launch will read, so
 * that its start does not wait on DRAM.  It is validated like `mats` (its
 * pointers must be device memory); nothing is written through it.
 * NVFP4 and MXFP4 run as one tensor-core launch, affine as one launch of the
 * affine GEMV, when the stacked rows have a plan and every scale (and bias)
 * row is 16-byte aligned; other cases run as mats->count qmv launches (and
 * ignore the hint).  Otherwise qmv's rules. */
fp4_status qmv_grouped(const fp4_bf16* x, const fp4_matrix_group* mats, fp4_mode mode, int bits, int group_size,
                       fp4_bf16* const* y, const fp4_matrix_group* prefetch_next, cudaStream_t stream);

/* qqmv: the one-row route of the quantized-activation matmul [P3 qqmm.cpp,
 * QQMatmul::eval_gpu: with quantized W and a single row of x, x goes through
 * fp_quantize_dequantize into an array of x's dtype and then through fp_qmv].
 *   y[n] = sum_k xhat[k] * deq(W)[n, k]   (fp32 accumulation, bf16 output)
 *   xhat = fp4_dequantize(fp4_quantize(x)): per block of 16 (NVFP4, global scale
 *          global_scale_x or 1) or 32 (MXFP4) the rule of fp4_quantize, then each
 *          value bf16_rn(fl(fl(e2m1(q) * scale) * gs_x)) -- x's own dtype, as the
 *          page's route stores it.  The quantization happens inside the GEMV
 *          kernel (no extra launch, no scratch).
 *   x, w, scales, global_scale_w, y, N, K: as for qmv (linear scales); mode is
 *          NVFP4 or MXFP4; global_scale_x (device fp32 or NULL) is NVFP4 only.
 * Requires K % 32 == 0 (hence whole blocks) and K <= 65536.  Launch order as qmv. */
fp4_status qqmv(const fp4_bf16* x, const float* global_scale_x, const uint32_t* w, const uint8_t* scales,
                const float* global_scale_w, int64_t N, int64_t K, fp4_mode mode, fp4_bf16* y,
                cudaStream_t stream);

/* a7-a9: qqmm, the FP4 x FP4 GEMM [P3 qqmm.cpp, qqmm_impl, qqmm_utils.cu].
 *   out[m, n] = bf16( alpha * sum_k deq(xq)[m, k] * deq(wq)[n, k] ),  beta = 0
 *   alpha = (*global_scale_x) * (*global_scale_w); a NULL pointer counts as 1.
 *   With multiplier-form global scales this is amax_x*amax_w/(448*6)^2.  To pass a
 *   precomputed alpha, give it as global_scale_x and NULL as global_scale_w.
 *   xq      uint32[M, K/8], 16-byte aligned (NVFP4 or MXFP4 codes)
 *   sx      uint8 block scales of xq, TILED_128x4 layout
 *   wq      uint32[N, K/8] (W stored [N, K]), 16-byte aligned
 *   sw      uint8 block scales of wq, TILED_128x4 layout
 *   out     bf16[M, N], 16-byte aligned
 * Requires K % 256 == 0 (hence K % 64 == 0 for the tensor-core K step), N % 8 == 0,
 * M >= 1.  mode is NVFP4 (E4M3 scales, group 16) or MXFP4 (E8M0, group 32). */
fp4_status qqmm(const uint32_t* xq, const uint8_t* sx, const uint32_t* wq, const uint8_t* sw,
                const float* global_scale_x, const float* global_scale_w, int64_t M, int64_t N,
                int64_t K, fp4_mode mode, fp4_bf16* out, cudaStream_t stream);

/* a10: gather_qmm, the MoE grouped GEMM with 4-bit weights and bf16 activations
 * [P2 Diagnosis 1 and 5: gather_gemm / grouped GEMM].
 *   out[r, n] = sum_k x[lhs_idx[r], k] * deq(w[rhs_idx[r]])[n, k]  (fp32 accumulation)
 *   x        bf16[T, K] activations (T = 1 + max lhs_idx), 16-byte aligned
 *   lhs_idx  int32[R] activation row of each routed row
 *   rhs_idx  int32[R] expert of each routed row, in [0, E)
 *   w        uint32[E, N, K/8], 16-byte aligned
 *   scales   MXFP4 uint8[E, N, K/32] E8M0, NVFP4 uint8[E, N, K/16] E4M3 (no global
 *            scale), affine bf16[E, N, K/group]; linear layout, 2-byte aligned
 *   biases   affine: bf16[E, N, K/group]; NULL otherwise
 *   out      bf16[R, N], 16-byte aligned
 * sorted != 0 promises rhs_idx is non-decreasing (rows grouped by expert), which
 * this version requires.  Requires K % 64 == 0 and N % 16 == 0.  The expert ids
 * live in device memory, so the kernel checks them: an id outside [0, E) or a
 * decrease leaves the affected output rows unwritten and makes the next
 * fp4_check_device_error return FP4_ERR_INVALID_ARG.  lhs_idx values must lie in
 * [0, T); they are not checked.  A tile whose routed rows are consecutive rows
 * of x (activations already in routed order, e.g. after gather_rows) loads
 * them by TMA; scattered rows are gathered 16 bytes at a time. */
fp4_status gather_qmm(const fp4_bf16* x, const int32_t* lhs_idx, const int32_t* rhs_idx, int64_t R,
                      const uint32_t* w, const void* scales, const fp4_bf16* biases, int64_t E,
                      int64_t N, int64_t K, fp4_mode mode, int bits, int group_size, int sorted,
                      fp4_bf16* out, cudaStream_t stream);

/* gather_rows: the routed activations in routing order [P2 Diagnosis 5: the
 * MoE grouped GEMM gathers each routed row's activations], so that a following
 * gather_qmm with lhs_idx = 0 .. R-1 reads them as whole tiles.
 *   out[i, :] = x[idx[i], :]   for i < R (pure data movement, bit-exact)
 *   x      bf16[x_rows, K], 16-byte aligned;  idx int32[R], 4-byte aligned
 *   out    bf16[R, K], 16-byte aligned, caller-owned (R K 2 bytes)
 * Requires K % 8 == 0.  An index outside [0, x_rows) leaves its output row
 * unwritten and makes the next fp4_check_device_error return
 * FP4_ERR_INVALID_ARG. */
fp4_status gather_rows(const fp4_bf16* x, int64_t x_rows, const int32_t* idx, int64_t R, int64_t K, fp4_bf16* out,
                       cudaStream_t stream);

/* qqmm_batched: batch_count independent FP4 x FP4 GEMMs in one launch [P3
 * qqmm_impl: the page's cuBLASLt call fixes the batch count at 1; this is the
 * strided-batch generalization].
 *   out_b = bf16( gs_x[b] * gs_w[b] * Xq_b . Wq_b^T ),  b = 0 .. batch - 1
 *   Xq_b = xq + b * stride_xq (uint32 words), its tiled scales sx + b * stride_sx (bytes);
 *   Wq_b = wq + b * stride_wq, scales sw + b * stride_sw; a stride of 0 shares one W
 *   (and its scales) across the batch; out_b = out + b * stride_out (elements).
 *   global_scale_x / global_scale_w: device fp32 arrays of `batch` values, or NULL (1).
 * Each batch follows qqmm's rules (M, N, K, layouts, alignment).  The strides
 * must keep the batches apart (stride_xq >= M K / 8, stride_sx >= the padded
 * scale bytes, stride_out >= M N, and likewise for W unless 0) and aligned
 * (16 bytes for codes and scales, 8 elements for out); batch <= 65535. */
fp4_status qqmm_batched(const uint32_t* xq, const uint8_t* sx, const uint32_t* wq, const uint8_t* sw,
                        const float* global_scale_x, const float* global_scale_w, int64_t batch, int64_t M,
                        int64_t N, int64_t K, int64_t stride_xq, int64_t stride_sx, int64_t stride_wq,
                        int64_t stride_sw, int64_t stride_out, fp4_mode mode, fp4_bf16* out, cudaStream_t stream);

/* Workspace bytes qqmm_quantize_x needs for an M x K activation. */
size_t qqmm_quantize_x_workspace_bytes(int64_t M, int64_t K, fp4_mode mode);

/* qqmm_quantize_x: the quantized-activation GEMM with the activation's
 * quantization fused into the same launch [P3 qqmm.cpp: QQMatmul::eval_gpu
 * quantizes x with quantize_input (fp_quantize, optional global scale) and then
 * calls the block-scaled GEMM -- separate launches there].
 *   out = bf16( gs_x * gs_w * fp4_quantize(x, gs_x) . Wq^T ), bit for bit what
 *   fp4_amax_global_scale (when global_scale_x is NULL) + fp4_quantize (tiled
 *   scales) + qqmm compute.
 *   x        bf16[M, K], 16-byte aligned
 *   global_scale_x  NVFP4: device fp32 activation global scale (a calibrated value),
 *            or NULL to take fl(amax(x) / 2688) from x; MXFP4: must be NULL
 *   global_scale_x_out  NVFP4 only, nullable: receives the activation scale used
 *   wq, sw, global_scale_w, M, N, K, mode, out: as for qqmm
 *   ws       device workspace of ws_bytes >= qqmm_quantize_x_workspace_bytes(M, K, mode)
 *            bytes, 128-byte aligned.  It must be zero-filled once when allocated;
 *            each call leaves its grid-barrier words ready for the next.  The
 *            quantized x (codes, then 128x4-tiled scales) sits at its start.
 *            Calls that overlap on the GPU must not share a workspace.
 * One persistent cooperative launch: every CTA quantizes a share of x (after a
 * grid-wide amax when NVFP4 has no activation scale), a grid barrier, then the
 * GEMM reads the quantized x from the workspace (still in L2).  The launch needs
 * every CTA resident (at most one per SM); a device that cannot co-schedule it
 * returns FP4_ERR_CUDA. */
fp4_status qqmm_quantize_x(const fp4_bf16* x, const float* global_scale_x, const uint32_t* wq, const uint8_t* sw,
                           const float* global_scale_w, int64_t M, int64_t N, int64_t K, fp4_mode mode, void* ws,
                           size_t ws_bytes, float* global_scale_x_out, fp4_bf16* out, cudaStream_t stream);

/* qmm: the dense prefill GEMM with 4-bit weights and bf16 activations (W4A16)
 * ["mlx: opt-in dense GEMM for nvfp4 prefill ... - #287": the mixed-input GEMM
 * of bf16 activations against NVFP4 weights at M > 1; "perf(cuda): enable
 * hardware NVFP4/MXFP4 conversion on Blackwell builds": qmm_sm80].
 *   out[m, n] = sum_k x[m, k] * deq(W)[n, k]   (fp32 accumulation, bf16 output)
 *   x        bf16[M, K], 16-byte aligned
 *   w        uint32[N, K/8] (W stored [N, K]), 16-byte aligned
 *   scales   linear block scales: NVFP4 uint8[N, K/16], MXFP4 uint8[N, K/32], affine
 *            bf16[N, K/group]; 2-byte aligned
 *   biases   affine: bf16[N, K/group]; NULL otherwise
 *   global_scale_w NVFP4 only: device fp32 gs of W (applied to the fp32 sums), or NULL
 *   out      bf16[M, N], 16-byte aligned
 * The weights are dequantized exactly (FP4: e2m1 * block scale is exact in bf16;
 * affine: q * scale + bias in fp32 carried as two bf16 terms).  Requires
 * K % 64 == 0 and N % 16 == 0. */
fp4_status qmm(const fp4_bf16* x, const uint32_t* w, const void* scales, const fp4_bf16* biases,
               const float* global_scale_w, int64_t M, int64_t N, int64_t K, fp4_mode mode, int bits, int group_size,
               fp4_bf16* out, cudaStream_t stream);

/* Maximum element count accepted by fp4_amax_global_scale_noalloc (2^36). */
#define FP4_AMAX_NOALLOC_MAX_ELEMS ((int64_t)1 << 36)

/* Allocation-free variant of fp4_amax_global_scale.  The pages have no
 * counterpart: this entry point exists for callers that cannot allocate device
 * memory where they need a global scale -- code recording into a CUDA stream
 * capture, engines that hand every kernel a pre-planned memory arena, hosts
 * that forbid allocation on a latency-critical path.  The per-block partial
 * maxima that fp4_amax_global_scale keeps in caller scratch live here in a
 * fixed 4 KiB file-scope device array (1024 partials) that every GPU loading
 * the library holds until the process exits.  The results are identical to
 * fp4_amax_global_scale's.
 *   x, n, gs_out, amax_out: as for fp4_amax_global_scale; n in [1, 2^36],
 *            larger n returns FP4_ERR_INVALID_ARG.
 * Nothing is allocated or freed, by this library or through any allocating
 * library routine.  The first call on a device looks up the array's device
 * address (cudaGetSymbolAddress) and checks the compute capability; make that
 * first call before any stream capture.  All calls share the array and it keeps
 * the last call's contents (each call writes every slot it reads, so nothing
 * needs clearing); calls that overlap on the GPU -- unordered streams -- race
 * on it and give unspecified results. */
fp4_status fp4_amax_global_scale_noalloc(const fp4_bf16* x, int64_t n, float* gs_out, float* amax_out,
                                         cudaStream_t stream);

/* Test hook, off by default: when `enable` is nonzero the next launches of the
 * tensor-core kernels -- qqmm, qmv's NVFP4/MXFP4 path and gather_qmm -- make
 * their MMA-issuing thread wait on a barrier nothing arrives at, with a 1 ms
 * limit, before doing their normal work.  The wait expires, the kernel records
 * FP4_ERR_TIMEOUT and still completes with a correct result; nothing faults or
 * hangs. */
fp4_status fp4_debug_inject_wait_timeout(int enable);

/* Measurement aid (no counterpart on the pages): moves NVFP4 weights from HBM
 * into shared memory exactly as qmv's tensor-core path streams them -- the same
 * split of K over CTAs, rows per CTA and ring of slots, one TMA box of R rows x
 * 128 bytes of codes and one of R rows x 16 bytes of scales per K = 256 stage,
 * programmatic dependent launch, consumption after the previous kernel -- and
 * computes nothing.  Timing it over the same weights as qmv gives the
 * launch-and-stream ceiling of that kernel shape.
 *   w       uint32[N, K/8], 16-byte aligned      scales  uint8[N, K/16], 16-byte aligned
 * Requires K % 256 == 0; a shape the tensor-core path does not take returns
 * FP4_ERR_UNSUPPORTED. */
fp4_status fp4_debug_stream_weights(const uint32_t* w, const uint8_t* scales, int64_t N, int64_t K,
                                    cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif
