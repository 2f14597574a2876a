// launch.h -- host-side launchers shared between the C ABI (api.cu) and the
// kernel translation units.  Arguments reaching these functions have already
// been validated by api.cu; each returns the cudaError_t of its launch(es).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

namespace fp4 {

struct DevInfo {
  int device = -1;
  int sm_count = 0;
  size_t smem_optin = 0;   // max dynamic shared memory per block (opt-in)
  unsigned* err = nullptr; // device address of the error word on this device
};

// api.cu: the current device's cached properties (initialized on first use);
// returns an fp4_status value
int current_device_info(const DevInfo** out);

// quant.cu
size_t amax_workspace_bytes(int64_t n);
cudaError_t launch_amax(const DevInfo& d, const uint16_t* x, int64_t n, float* gs_out,
                        float* amax_out, uint32_t* partials, int max_partials, cudaStream_t s);
// sr != 0: stochastic rounding of the elements (Philox4x32-10 words from seed and offset)
cudaError_t launch_quantize(const DevInfo& d, const uint16_t* x, int64_t rows, int64_t cols,
                            int mode, int group, const float* gs, uint32_t* xq, uint8_t* scales,
                            int tiled, int sr, uint64_t seed, uint64_t offset, cudaStream_t s);
cudaError_t launch_dequantize(const DevInfo& d, const uint32_t* wq, const void* scales,
                              const uint16_t* biases, int64_t rows, int64_t cols, int mode,
                              int group, const float* gs, int tiled, uint16_t* out,
                              cudaStream_t s);

// qmv.cu (qx != 0: the quantized-activation route -- x is replaced by
// fp_dequantize(fp_quantize(x, gs_x)) before the GEMV; NVFP4 and MXFP4 only)
cudaError_t launch_qmv(const DevInfo& d, const uint16_t* x, const float* gs_x, int qx, const uint32_t* w,
                       const void* scales, const uint16_t* biases, const float* gs_w, int64_t N, int64_t K,
                       int mode, int group, uint16_t* y, int inject_timeout, cudaStream_t s);

// qmv_tc.cu (NVFP4 = mode 2 and MXFP4 = mode 1 on tcgen05; launch_qmv dispatches to it when supported)
PFN_cuTensorMapEncodeTiled_v12000 encode_fn();  // driver's tensor-map encoder (nullptr if unavailable)
// the NVFP4 plan: CTAs per cluster (K slices), row blocks, rows per CTA, weight ring slots
bool qmv_tc_geometry(const DevInfo& d, int64_t N, int64_t K, int* split, int* nblk, int* R, int* nslots);
bool qmv_tc_supported(const DevInfo& d, int mode, int64_t N, int64_t K);
bool qmv_tc_group_supported(const DevInfo& d, int mode, int count, const int64_t* N, int64_t K);
// the weights of a GEMV launch (a group of up to 4 matrices of one K)
struct GemvGroupDesc {
  int count = 0;
  const uint32_t* w[4] = {};
  const uint8_t* scales[4] = {};   // FP4: E4M3/E8M0 bytes; affine: bf16 scales
  const uint16_t* biases[4] = {};  // affine only
  int64_t N[4] = {};
  int64_t K = 0;
};
cudaError_t launch_qmv_tc_group(const DevInfo& d, int mode, const uint16_t* x, const float* gs_x, int qx, int count,
                                const uint32_t* const* w, const uint8_t* const* scales, const float* const* gs_w,
                                const int64_t* N, int64_t K, uint16_t* const* y, const GemvGroupDesc* next,
                                int inject_timeout, cudaStream_t s);
cudaError_t launch_qmv_tc(const DevInfo& d, int mode, const uint16_t* x, const float* gs_x, int qx,
                          const uint32_t* w, const uint8_t* scales, const float* gs_w, int64_t N, int64_t K,
                          uint16_t* y, int inject_timeout, cudaStream_t s);

// qmv_affine.cu (affine-4 GEMV on a TMA ring; launch_qmv dispatches to it when the plan fits:
// K a multiple of max(512, 8 group) and at most 32768, 16-byte aligned scales and biases)
bool qmv_affine_supported(const DevInfo& d, int64_t N, int64_t K, int group);
cudaError_t launch_qmv_affine(const DevInfo& d, const uint16_t* x, const uint32_t* w, const uint16_t* scales,
                              const uint16_t* biases, int64_t N, int64_t K, int group, uint16_t* y,
                              cudaStream_t s);
bool qmv_affine_group_supported(const DevInfo& d, int count, const int64_t* N, int64_t K, int group);
cudaError_t launch_qmv_affine_group(const DevInfo& d, const uint16_t* x, int count, const uint32_t* const* w,
                                    const uint16_t* const* scales, const uint16_t* const* biases, const int64_t* N,
                                    int64_t K, int group, uint16_t* const* y, const GemvGroupDesc* next,
                                    cudaStream_t s);

// qqmm.cu: batch b reads xq + b stride_xq (uint32 words), sx + b stride_sx (bytes),
// wq + b stride_wq (0: one W for every batch), sw + b stride_sw, gs_x[b], gs_w[b],
// and writes out + b stride_out (elements); a plain call is batch 1.
struct BatchArgs {
  int64_t batch = 1;
  int64_t stride_xq = 0, stride_sx = 0, stride_wq = 0, stride_sw = 0, stride_out = 0;
};
cudaError_t launch_qqmm(const DevInfo& d, const uint32_t* xq, const uint8_t* sx, const uint32_t* wq,
                        const uint8_t* sw, const float* gs_x, const float* gs_w, int64_t M,
                        int64_t N, int64_t K, const BatchArgs& ba, int mode, uint16_t* out, int inject_timeout,
                        cudaStream_t s);

// qqmm.cu: the fused call -- bf16 x quantized by the same (cooperative) launch
// into the workspace, then the GEMM (gs_in: the NVFP4 activation global scale,
// or nullptr to take amax(x) / 2688; gs_out: where the scale used goes, nullable)
size_t qqmm_fused_workspace_bytes(int64_t M, int64_t K, int mode);
cudaError_t launch_qqmm_fused(const DevInfo& d, const uint16_t* x, const float* gs_in, float* gs_out,
                              const uint32_t* wq, const uint8_t* sw, const float* gs_w, int64_t M, int64_t N,
                              int64_t K, int mode, void* ws, uint16_t* out, int inject_timeout, cudaStream_t s);

// weight_stream.cu (measurement aid: the GEMV's weight stream without the GEMV)
cudaError_t launch_weight_stream(const DevInfo& d, const uint32_t* w, const uint8_t* scales, int64_t N,
                                 int64_t K, cudaStream_t s);

// gather_qmm.cu: W4A16 GEMMs (MXFP4 = 1, NVFP4 = 2, affine = 0 weights) -- the MoE
// gather_qmm (rows sorted by expert) and the dense qmm (gs_w: NVFP4 weight global
// scale or nullptr; biases: affine only)
cudaError_t launch_gather_rows(const DevInfo& d, const uint16_t* x, int64_t x_rows, const int32_t* idx, int64_t R,
                               int64_t K, uint16_t* out, cudaStream_t s);
cudaError_t launch_gather_qmm(const DevInfo& d, const uint16_t* x, const int32_t* lhs, const int32_t* rhs, int64_t R,
                              const uint32_t* w, const void* scales, const uint16_t* biases, const float* gs_w,
                              int64_t E, int64_t N, int64_t K, int mode, int group, uint16_t* out, int inject_timeout,
                              cudaStream_t s);
cudaError_t launch_qmm(const DevInfo& d, const uint16_t* x, int64_t M, const uint32_t* w, const void* scales,
                       const uint16_t* biases, const float* gs_w, int64_t N, int64_t K, int mode, int group,
                       uint16_t* out, int inject_timeout, cudaStream_t s);

}  // namespace fp4
