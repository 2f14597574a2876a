// api.cu -- the C ABI of libfp4gb300: host-side validation, per-device state
// and launches.  No entry point throws, allocates or keeps a pointer.
#include <atomic>
#include <cstdio>
#include <mutex>

#include "../../include/fp4_gb300.h"
#include "common.cuh"
#include "launch.h"

namespace fp4 {
namespace {

// Device error word, one per device context.  Bounded waits that expire
// atomically OR kErrTimeout into it, index checks kErrIndex;
// fp4_check_device_error reads and clears it.
__device__ unsigned g_device_error;

constexpr int kMaxDevices = 64;
DevInfo g_dev[kMaxDevices];
std::mutex g_mu;
std::atomic<int> g_inject_timeout{0};

fp4_status init_device(int device, const DevInfo** out) {
  if (device < 0 || device >= kMaxDevices) return FP4_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mu);
  DevInfo& d = g_dev[device];
  if (d.device == device) {
    *out = &d;
    return FP4_OK;
  }
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return FP4_ERR_CUDA;
  if (prop.major != 10 || prop.minor != 3) return FP4_ERR_UNSUPPORTED;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return FP4_ERR_CUDA;
  if (cur != device && cudaSetDevice(device) != cudaSuccess) return FP4_ERR_CUDA;
  void* err_addr = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&err_addr, g_device_error);
  if (e == cudaSuccess) e = cudaMemset(err_addr, 0, sizeof(unsigned));
  if (cur != device) cudaSetDevice(cur);
  if (e != cudaSuccess) return FP4_ERR_CUDA;
  d.sm_count = prop.multiProcessorCount;
  d.smem_optin = prop.sharedMemPerBlockOptin;
  d.err = static_cast<unsigned*>(err_addr);
  d.device = device;
  *out = &d;
  return FP4_OK;
}

fp4_status current(const DevInfo** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return FP4_ERR_CUDA;
  return init_device(dev, out);
}

}  // namespace

int current_device_info(const DevInfo** out) { return (int)current(out); }

namespace {

fp4_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return FP4_OK;
  if (e == cudaErrorInvalidValue) return FP4_ERR_INVALID_ARG;
  return FP4_ERR_CUDA;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// mode/bits/group combinations of the pages: affine 4-bit groups 32/64/128,
// MXFP4 4-bit group 32, NVFP4 4-bit group 16.
fp4_status check_format(int mode, int bits, int group) {
  if (bits != 4) return FP4_ERR_UNSUPPORTED;
  if (mode == FP4_MODE_NVFP4) return group == 16 ? FP4_OK : FP4_ERR_UNSUPPORTED;
  if (mode == FP4_MODE_MXFP4) return group == 32 ? FP4_OK : FP4_ERR_UNSUPPORTED;
  if (mode == FP4_MODE_AFFINE)
    return (group == 32 || group == 64 || group == 128) ? FP4_OK : FP4_ERR_UNSUPPORTED;
  return FP4_ERR_UNSUPPORTED;
}

}  // namespace
}  // namespace fp4

using namespace fp4;

extern "C" {

fp4_status fp4_init(int device) {
  const DevInfo* d = nullptr;
  return init_device(device, &d);
}

const char* fp4_status_string(fp4_status s) {
  switch (s) {
    case FP4_OK: return "ok";
    case FP4_ERR_INVALID_ARG: return "invalid argument";
    case FP4_ERR_UNSUPPORTED: return "unsupported mode/bits/group combination or device";
    case FP4_ERR_ALIGNMENT: return "pointer or row pitch misaligned";
    case FP4_ERR_CUDA: return "CUDA runtime error";
    case FP4_ERR_TIMEOUT: return "a bounded device wait expired";
  }
  return "unknown status";
}

fp4_status fp4_check_device_error(cudaStream_t stream) {
  const DevInfo* d = nullptr;
  fp4_status st = current(&d);
  if (st != FP4_OK) return st;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return FP4_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpy(&v, d->err, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return FP4_ERR_CUDA;
  if (v != 0) {
    const unsigned zero = 0;
    if (cudaMemcpy(d->err, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return FP4_ERR_CUDA;
    return (v & kErrTimeout) ? FP4_ERR_TIMEOUT : FP4_ERR_INVALID_ARG;
  }
  return FP4_OK;
}

void fp4_padded_scale_dims(int64_t rows, int64_t scale_cols, int64_t* padded_rows, int64_t* padded_cols) {
  if (padded_rows) *padded_rows = ((rows + 127) / 128) * 128;
  if (padded_cols) *padded_cols = ((scale_cols + 3) / 4) * 4;
}

size_t fp4_amax_workspace_bytes(int64_t n) { return amax_workspace_bytes(n); }

fp4_status fp4_amax_global_scale(const fp4_bf16* x, int64_t n, float* gs_out, float* amax_out, void* ws,
                                 size_t ws_bytes, cudaStream_t stream) {
  if (!x || !gs_out || !ws || n <= 0) return FP4_ERR_INVALID_ARG;
  if (ws_bytes < amax_workspace_bytes(n)) return FP4_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(gs_out, 4) || !aligned(ws, 4) || (amax_out && !aligned(amax_out, 4)))
    return FP4_ERR_ALIGNMENT;
  const DevInfo* d = nullptr;
  fp4_status st = current(&d);
  if (st != FP4_OK) return st;
  const int max_partials = (int)(ws_bytes / sizeof(uint32_t));
  return from_cuda(launch_amax(*d, x, n, gs_out, amax_out, static_cast<uint32_t*>(ws),
                               max_partials > 1024 ? 1024 : max_partials, stream));
}

namespace {
fp4_status quantize_common(const fp4_bf16* x, int64_t rows, int64_t cols, fp4_mode mode, int bits, int group_size,
                           const float* global_scale, uint32_t* xq, uint8_t* scales, fp4_scale_layout layout,
                           int sr, uint64_t seed, uint64_t offset, cudaStream_t stream) {
  fp4_status st = check_format(mode, bits, group_size);
  if (st != FP4_OK) return st;
  if (mode == FP4_MODE_AFFINE) return FP4_ERR_UNSUPPORTED;
  if (!x || !xq || !scales || rows <= 0 || cols <= 0) return FP4_ERR_INVALID_ARG;
  if (cols % group_size != 0) return FP4_ERR_INVALID_ARG;
  if (rows > INT32_MAX / 2 || cols > INT32_MAX / 16) return FP4_ERR_INVALID_ARG;
  if (global_scale && mode != FP4_MODE_NVFP4) return FP4_ERR_INVALID_ARG;
  if (layout != FP4_SCALES_LINEAR && layout != FP4_SCALES_TILED_128x4) return FP4_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(xq, mode == FP4_MODE_NVFP4 ? 8 : 16) ||
      (global_scale && !aligned(global_scale, 4)))
    return FP4_ERR_ALIGNMENT;
  const DevInfo* d = nullptr;
  st = current(&d);
  if (st != FP4_OK) return st;
  return from_cuda(launch_quantize(*d, x, rows, cols, mode, group_size, global_scale, xq, scales,
                                   layout == FP4_SCALES_TILED_128x4, sr, seed, offset, stream));
}
}  // namespace

fp4_status fp4_quantize(const fp4_bf16* x, int64_t rows, int64_t cols, fp4_mode mode, int bits,
                        int group_size, const float* global_scale, uint32_t* xq, uint8_t* scales,
                        fp4_scale_layout layout, cudaStream_t stream) {
  return quantize_common(x, rows, cols, mode, bits, group_size, global_scale, xq, scales, layout, 0, 0, 0, stream);
}

fp4_status fp4_quantize_sr(const fp4_bf16* x, int64_t rows, int64_t cols, fp4_mode mode, int bits,
                           int group_size, const float* global_scale, uint64_t seed, uint64_t offset, uint32_t* xq,
                           uint8_t* scales, fp4_scale_layout layout, cudaStream_t stream) {
  return quantize_common(x, rows, cols, mode, bits, group_size, global_scale, xq, scales, layout, 1, seed, offset,
                         stream);
}

fp4_status fp4_dequantize(const uint32_t* wq, const void* scales, const fp4_bf16* biases, int64_t rows,
                          int64_t cols, fp4_mode mode, int bits, int group_size, const float* global_scale,
                          fp4_scale_layout layout, fp4_bf16* out, cudaStream_t stream) {
  fp4_status st = check_format(mode, bits, group_size);
  if (st != FP4_OK) return st;
  if (!wq || !scales || !out || rows <= 0 || cols <= 0 || cols % group_size != 0) return FP4_ERR_INVALID_ARG;
  if (mode == FP4_MODE_AFFINE) {
    if (!biases || layout != FP4_SCALES_LINEAR || global_scale) return FP4_ERR_INVALID_ARG;
    if (!aligned(scales, 2) || !aligned(biases, 2)) return FP4_ERR_ALIGNMENT;
  } else {
    if (biases) return FP4_ERR_INVALID_ARG;
    if (global_scale && mode != FP4_MODE_NVFP4) return FP4_ERR_INVALID_ARG;
    if (layout != FP4_SCALES_LINEAR && layout != FP4_SCALES_TILED_128x4) return FP4_ERR_INVALID_ARG;
  }
  if (!aligned(wq, 4) || !aligned(out, 16) || (global_scale && !aligned(global_scale, 4))) return FP4_ERR_ALIGNMENT;
  const DevInfo* d = nullptr;
  st = current(&d);
  if (st != FP4_OK) return st;
  return from_cuda(launch_dequantize(*d, wq, scales, biases, rows, cols, mode, group_size, global_scale,
                                     layout == FP4_SCALES_TILED_128x4, out, stream));
}

fp4_status qmv(const fp4_bf16* x, const uint32_t* w, const void* scales, const fp4_bf16* biases,
               const float* global_scale_w, int64_t N, int64_t K, fp4_mode mode, int bits, int group_size,
               fp4_bf16* y, cudaStream_t stream) {
  fp4_status st = check_format(mode, bits, group_size);
  if (st != FP4_OK) return st;
  if (!x || !w || !scales || !y || N <= 0 || K <= 0) return FP4_ERR_INVALID_ARG;
  if (K % 32 != 0 || K % group_size != 0 || N > INT32_MAX / 2) return FP4_ERR_INVALID_ARG;
  if (K > 65536) return FP4_ERR_UNSUPPORTED;  // x is staged whole in shared memory
  if (mode == FP4_MODE_AFFINE) {
    if (!biases || global_scale_w) return FP4_ERR_INVALID_ARG;
    if (!aligned(scales, 2) || !aligned(biases, 2)) return FP4_ERR_ALIGNMENT;
  } else {
    if (biases) return FP4_ERR_INVALID_ARG;
    if (global_scale_w && mode != FP4_MODE_NVFP4) return FP4_ERR_INVALID_ARG;
    if (mode == FP4_MODE_NVFP4 && !aligned(scales, 2)) return FP4_ERR_ALIGNMENT;
  }
  if (!aligned(x, 16) || !aligned(w, 16) || !aligned(y, 2)) return FP4_ERR_ALIGNMENT;
  const DevInfo* d = nullptr;
  st = current(&d);
  if (st != FP4_OK) return st;
  return from_cuda(launch_qmv(*d, x, nullptr, 0, w, scales, biases, global_scale_w, N, K, mode, group_size, y,
                              g_inject_timeout.load(), stream));
}

namespace {
// one group of qmv_grouped: each matrix a valid qmv on its own (same checks, same x)
fp4_status check_group(const fp4_bf16* x, const fp4_matrix_group* g, fp4_mode mode, int bits, int group_size) {
  if (!g || g->count < 1 || g->count > 4) return FP4_ERR_INVALID_ARG;
  fp4_status st = check_format(mode, bits, group_size);
  if (st != FP4_OK) return st;
  const int64_t K = g->K;
  if (!x || K <= 0 || K % 32 != 0 || K % group_size != 0) return FP4_ERR_INVALID_ARG;
  if (K > 65536) return FP4_ERR_UNSUPPORTED;
  for (int i = 0; i < g->count; ++i) {
    if (!g->w[i] || !g->scales[i] || g->N[i] <= 0 || g->N[i] > INT32_MAX / 2) return FP4_ERR_INVALID_ARG;
    const fp4_bf16* b = g->biases[i];
    const float* gs = g->global_scale_w[i];
    if (mode == FP4_MODE_AFFINE) {
      if (!b || gs) return FP4_ERR_INVALID_ARG;
      if (!aligned(g->scales[i], 2) || !aligned(b, 2)) return FP4_ERR_ALIGNMENT;
    } else {
      if (b) return FP4_ERR_INVALID_ARG;
      if (gs && mode != FP4_MODE_NVFP4) return FP4_ERR_INVALID_ARG;
      if (gs && !aligned(gs, 4)) return FP4_ERR_ALIGNMENT;
      if (mode == FP4_MODE_NVFP4 && !aligned(g->scales[i], 2)) return FP4_ERR_ALIGNMENT;
    }
    if (!aligned(x, 16) || !aligned(g->w[i], 16)) return FP4_ERR_ALIGNMENT;
  }
  return FP4_OK;
}

// whether the tensor-core GEMV takes the whole group in one launch
bool group_on_tc(const DevInfo& d, const fp4_matrix_group* g, fp4_mode mode) {
  if (mode != FP4_MODE_NVFP4 && mode != FP4_MODE_MXFP4) return false;
  for (int i = 0; i < g->count; ++i)
    if (!aligned(g->scales[i], 16)) return false;
  return qmv_tc_group_supported(d, mode, g->count, g->N, g->K);
}

// whether the affine TMA GEMV takes the whole group in one launch
bool group_on_affine(const DevInfo& d, const fp4_matrix_group* g, fp4_mode mode, int group_size) {
  if (mode != FP4_MODE_AFFINE) return false;
  for (int i = 0; i < g->count; ++i)
    if (!aligned(g->scales[i], 16) || !aligned(g->biases[i], 16)) return false;
  return qmv_affine_group_supported(d, g->count, g->N, g->K, group_size);
}

void fill_desc(const fp4_matrix_group* g, GemvGroupDesc* nd) {
  nd->count = g->count;
  nd->K = g->K;
  for (int i = 0; i < g->count; ++i) {
    nd->w[i] = g->w[i];
    nd->scales[i] = static_cast<const uint8_t*>(g->scales[i]);
    nd->biases[i] = reinterpret_cast<const uint16_t*>(g->biases[i]);
    nd->N[i] = g->N[i];
  }
}
}  // namespace

fp4_status qmv_grouped(const fp4_bf16* x, const fp4_matrix_group* mats, fp4_mode mode, int bits, int group_size,
                       fp4_bf16* const* y, const fp4_matrix_group* prefetch_next, cudaStream_t stream) {
  fp4_status st = check_group(x, mats, mode, bits, group_size);
  if (st != FP4_OK) return st;
  if (!y) return FP4_ERR_INVALID_ARG;
  for (int i = 0; i < mats->count; ++i) {
    if (!y[i]) return FP4_ERR_INVALID_ARG;
    if (!aligned(y[i], 2)) return FP4_ERR_ALIGNMENT;
  }
  if (prefetch_next) {  // the hint is checked as strictly as the group itself
    st = check_group(x, prefetch_next, mode, bits, group_size);
    if (st != FP4_OK) return st;
  }
  const DevInfo* d = nullptr;
  st = current(&d);
  if (st != FP4_OK) return st;
  if (group_on_tc(*d, mats, mode)) {
    const uint8_t* sc[4];
    uint16_t* yy[4];
    for (int i = 0; i < mats->count; ++i) {
      sc[i] = static_cast<const uint8_t*>(mats->scales[i]);
      yy[i] = reinterpret_cast<uint16_t*>(y[i]);
    }
    GemvGroupDesc nd;
    const bool hint = prefetch_next && group_on_tc(*d, prefetch_next, mode);
    if (hint) fill_desc(prefetch_next, &nd);
    return from_cuda(launch_qmv_tc_group(*d, mode, x, nullptr, 0, mats->count, mats->w, sc, mats->global_scale_w,
                                         mats->N, mats->K, yy, hint ? &nd : nullptr, g_inject_timeout.load(),
                                         stream));
  }
  if (group_on_affine(*d, mats, mode, group_size)) {
    const uint16_t* sc[4];
    const uint16_t* bi[4];
    uint16_t* yy[4];
    for (int i = 0; i < mats->count; ++i) {
      sc[i] = static_cast<const uint16_t*>(mats->scales[i]);
      bi[i] = reinterpret_cast<const uint16_t*>(mats->biases[i]);
      yy[i] = reinterpret_cast<uint16_t*>(y[i]);
    }
    GemvGroupDesc nd;
    const bool hint = prefetch_next && group_on_affine(*d, prefetch_next, mode, group_size);
    if (hint) fill_desc(prefetch_next, &nd);
    return from_cuda(launch_qmv_affine_group(*d, x, mats->count, mats->w, sc, bi, mats->N, mats->K, group_size, yy,
                                             hint ? &nd : nullptr, stream));
  }
  for (int i = 0; i < mats->count; ++i) {
    const cudaError_t e = launch_qmv(*d, x, nullptr, 0, mats->w[i], mats->scales[i], mats->biases[i],
                                     mats->global_scale_w[i], mats->N[i], mats->K, mode, group_size, y[i],
                                     g_inject_timeout.load(), stream);
    if (e != cudaSuccess) return from_cuda(e);
  }
  return FP4_OK;
}

fp4_status qqmv(const fp4_bf16* x, const float* global_scale_x, const uint32_t* w, const uint8_t* scales,
                const float* global_scale_w, int64_t N, int64_t K, fp4_mode mode, fp4_bf16* y,
                cudaStream_t stream) {
  if (mode != FP4_MODE_NVFP4 && mode != FP4_MODE_MXFP4) return FP4_ERR_UNSUPPORTED;
  const int group = mode == FP4_MODE_NVFP4 ? 16 : 32;
  if (!x || !w || !scales || !y || N <= 0 || K <= 0) return FP4_ERR_INVALID_ARG;
  if (K % 32 != 0 || N > INT32_MAX / 2) return FP4_ERR_INVALID_ARG;
  if (K > 65536) return FP4_ERR_UNSUPPORTED;  // x is staged whole in shared memory
  if ((global_scale_x || global_scale_w) && mode != FP4_MODE_NVFP4) return FP4_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(w, 16) || !aligned(y, 2) || (mode == FP4_MODE_NVFP4 && !aligned(scales, 2)) ||
      (global_scale_x && !aligned(global_scale_x, 4)) || (global_scale_w && !aligned(global_scale_w, 4)))
    return FP4_ERR_ALIGNMENT;
  const DevInfo* d = nullptr;
  fp4_status st = current(&d);
  if (st != FP4_OK) return st;
  return from_cuda(launch_qmv(*d, x, global_scale_x, 1, w, scales, nullptr, global_scale_w, N, K, mode, group, y,
                              g_inject_timeout.load(), stream));
}

namespace {
fp4_status qqmm_common(const uint32_t* xq, const uint8_t* sx, const uint32_t* wq, const uint8_t* sw,
                       const float* global_scale_x, const float* global_scale_w, int64_t M, int64_t N, int64_t K,
                       const BatchArgs& ba, fp4_mode mode, fp4_bf16* out, cudaStream_t stream) {
  if (mode != FP4_MODE_NVFP4 && mode != FP4_MODE_MXFP4) return FP4_ERR_UNSUPPORTED;
  if (!xq || !sx || !wq || !sw || !out || M <= 0 || N <= 0 || K <= 0) return FP4_ERR_INVALID_ARG;
  if (K % 256 != 0 || N % 8 != 0 || M > INT32_MAX / 2 || N > INT32_MAX / 2 || K > (1 << 24))
    return FP4_ERR_INVALID_ARG;
  if (ba.batch < 1 || ba.batch > 65535) return FP4_ERR_INVALID_ARG;
  if (ba.batch > 1) {
    const int group = mode == FP4_MODE_NVFP4 ? 16 : 32;
    int64_t prm = 0, pcm = 0, prn = 0, pcn = 0;
    fp4_padded_scale_dims(M, K / group, &prm, &pcm);
    fp4_padded_scale_dims(N, K / group, &prn, &pcn);
    // every batch's operands lie apart (W and its scales may be shared: stride 0)
    if (ba.stride_xq < M * (K / 8) || ba.stride_sx < prm * pcm || ba.stride_out < M * N) return FP4_ERR_INVALID_ARG;
    if ((ba.stride_wq != 0 && ba.stride_wq < N * (K / 8)) || (ba.stride_sw != 0 && ba.stride_sw < prn * pcn))
      return FP4_ERR_INVALID_ARG;
    if (ba.stride_xq % 4 || ba.stride_wq % 4 || ba.stride_sx % 16 || ba.stride_sw % 16 || ba.stride_out % 8)
      return FP4_ERR_ALIGNMENT;
  }
  if (!aligned(xq, 16) || !aligned(wq, 16) || !aligned(sx, 16) || !aligned(sw, 16) || !aligned(out, 16))
    return FP4_ERR_ALIGNMENT;
  if ((global_scale_x && !aligned(global_scale_x, 4)) || (global_scale_w && !aligned(global_scale_w, 4)))
    return FP4_ERR_ALIGNMENT;
  const DevInfo* d = nullptr;
  fp4_status st = current(&d);
  if (st != FP4_OK) return st;
  return from_cuda(launch_qqmm(*d, xq, sx, wq, sw, global_scale_x, global_scale_w, M, N, K, ba, mode, out,
                               g_inject_timeout.load(), stream));
}
}  // namespace

fp4_status qqmm(const uint32_t* xq, const uint8_t* sx, const uint32_t* wq, const uint8_t* sw,
                const float* global_scale_x, const float* global_scale_w, int64_t M, int64_t N, int64_t K,
                fp4_mode mode, fp4_bf16* out, cudaStream_t stream) {
  return qqmm_common(xq, sx, wq, sw, global_scale_x, global_scale_w, M, N, K, BatchArgs{}, mode, out, stream);
}

fp4_status qqmm_batched(const uint32_t* xq, const uint8_t* sx, const uint32_t* wq, const uint8_t* sw,
                        const float* global_scale_x, const float* global_scale_w, int64_t batch, int64_t M,
                        int64_t N, int64_t K, int64_t stride_xq, int64_t stride_sx, int64_t stride_wq,
                        int64_t stride_sw, int64_t stride_out, fp4_mode mode, fp4_bf16* out, cudaStream_t stream) {
  BatchArgs ba;
  ba.batch = batch;
  ba.stride_xq = stride_xq;
  ba.stride_sx = stride_sx;
  ba.stride_wq = stride_wq;
  ba.stride_sw = stride_sw;
  ba.stride_out = stride_out;
  return qqmm_common(xq, sx, wq, sw, global_scale_x, global_scale_w, M, N, K, ba, mode, out, stream);
}

size_t qqmm_quantize_x_workspace_bytes(int64_t M, int64_t K, fp4_mode mode) {
  if (M <= 0 || K <= 0) return 0;
  return qqmm_fused_workspace_bytes(M, K, mode == FP4_MODE_NVFP4 ? 2 : 1);
}

fp4_status qqmm_quantize_x(const fp4_bf16* x, const float* global_scale_x, const uint32_t* wq, const uint8_t* sw,
                           const float* global_scale_w, int64_t M, int64_t N, int64_t K, fp4_mode mode, void* ws,
                           size_t ws_bytes, float* global_scale_x_out, fp4_bf16* out, cudaStream_t stream) {
  if (mode != FP4_MODE_NVFP4 && mode != FP4_MODE_MXFP4) return FP4_ERR_UNSUPPORTED;
  if (!x || !wq || !sw || !out || !ws || M <= 0 || N <= 0 || K <= 0) return FP4_ERR_INVALID_ARG;
  if (K % 256 != 0 || N % 8 != 0 || M > INT32_MAX / 2 || N > INT32_MAX / 2 || K > (1 << 24))
    return FP4_ERR_INVALID_ARG;
  if (mode == FP4_MODE_MXFP4 && (global_scale_x || global_scale_w || global_scale_x_out)) return FP4_ERR_INVALID_ARG;
  if (ws_bytes < qqmm_fused_workspace_bytes(M, K, mode == FP4_MODE_NVFP4 ? 2 : 1)) return FP4_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(wq, 16) || !aligned(sw, 16) || !aligned(out, 16) || !aligned(ws, 128) ||
      (global_scale_x && !aligned(global_scale_x, 4)) || (global_scale_w && !aligned(global_scale_w, 4)) ||
      (global_scale_x_out && !aligned(global_scale_x_out, 4)))
    return FP4_ERR_ALIGNMENT;
  const DevInfo* d = nullptr;
  fp4_status st = current(&d);
  if (st != FP4_OK) return st;
  return from_cuda(launch_qqmm_fused(*d, x, global_scale_x, global_scale_x_out, wq, sw, global_scale_w, M, N, K,
                                     mode == FP4_MODE_NVFP4 ? 2 : 1, ws, out, g_inject_timeout.load(), stream));
}

namespace {
// Shared checks of the W4A16 GEMMs: format, weight scales/biases by mode, alignment.
fp4_status check_w4a16(const fp4_bf16* x, const uint32_t* w, const void* scales, const fp4_bf16* biases,
                       const float* gs_w, fp4_mode mode, int bits, int group_size, int64_t N, int64_t K,
                       const fp4_bf16* out) {
  fp4_status st = check_format(mode, bits, group_size);
  if (st != FP4_OK) return st;
  if (!x || !w || !scales || !out) return FP4_ERR_INVALID_ARG;
  if (N <= 0 || K <= 0 || K % 64 != 0 || N % 16 != 0 || N > INT32_MAX / 2 || K > (1 << 20)) return FP4_ERR_INVALID_ARG;
  if ((mode == FP4_MODE_AFFINE) != (biases != nullptr)) return FP4_ERR_INVALID_ARG;
  if (gs_w && mode != FP4_MODE_NVFP4) return FP4_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(w, 16) || !aligned(out, 16) || !aligned(scales, 2) ||
      (biases && !aligned(biases, 2)) || (gs_w && !aligned(gs_w, 4)))
    return FP4_ERR_ALIGNMENT;
  return FP4_OK;
}
}  // namespace

fp4_status gather_qmm(const fp4_bf16* x, const int32_t* lhs_idx, const int32_t* rhs_idx, int64_t R,
                      const uint32_t* w, const void* scales, const fp4_bf16* biases, int64_t E, int64_t N,
                      int64_t K, fp4_mode mode, int bits, int group_size, int sorted, fp4_bf16* out,
                      cudaStream_t stream) {
  fp4_status st = check_w4a16(x, w, scales, biases, nullptr, mode, bits, group_size, N, K, out);
  if (st != FP4_OK) return st;
  if (!sorted) return FP4_ERR_UNSUPPORTED;
  if (!lhs_idx || !rhs_idx) return FP4_ERR_INVALID_ARG;
  if (R <= 0 || E <= 0 || R > INT32_MAX / 2 || E > 4096) return FP4_ERR_INVALID_ARG;
  if (!aligned(lhs_idx, 4) || !aligned(rhs_idx, 4)) return FP4_ERR_ALIGNMENT;
  const DevInfo* d = nullptr;
  st = current(&d);
  if (st != FP4_OK) return st;
  return from_cuda(launch_gather_qmm(*d, x, lhs_idx, rhs_idx, R, w, scales, biases, nullptr, E, N, K, mode,
                                     group_size, out, g_inject_timeout.load(), stream));
}

fp4_status gather_rows(const fp4_bf16* x, int64_t x_rows, const int32_t* idx, int64_t R, int64_t K, fp4_bf16* out,
                       cudaStream_t stream) {
  if (!x || !idx || !out || x_rows <= 0 || R <= 0 || K <= 0 || K % 8 != 0) return FP4_ERR_INVALID_ARG;
  if (R > INT32_MAX || x_rows > INT32_MAX || K > (1 << 24)) return FP4_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(out, 16) || !aligned(idx, 4)) return FP4_ERR_ALIGNMENT;
  const DevInfo* d = nullptr;
  fp4_status st = current(&d);
  if (st != FP4_OK) return st;
  return from_cuda(launch_gather_rows(*d, x, x_rows, idx, R, K, out, stream));
}

fp4_status qmm(const fp4_bf16* x, const uint32_t* w, const void* scales, const fp4_bf16* biases,
               const float* global_scale_w, int64_t M, int64_t N, int64_t K, fp4_mode mode, int bits, int group_size,
               fp4_bf16* out, cudaStream_t stream) {
  fp4_status st = check_w4a16(x, w, scales, biases, global_scale_w, mode, bits, group_size, N, K, out);
  if (st != FP4_OK) return st;
  if (M <= 0 || M > INT32_MAX / 2) return FP4_ERR_INVALID_ARG;
  const DevInfo* d = nullptr;
  st = current(&d);
  if (st != FP4_OK) return st;
  return from_cuda(launch_qmm(*d, x, M, w, scales, biases, global_scale_w, N, K, mode, group_size, out,
                              g_inject_timeout.load(), stream));
}

fp4_status fp4_debug_stream_weights(const uint32_t* w, const uint8_t* scales, int64_t N, int64_t K,
                                    cudaStream_t stream) {
  if (!w || !scales || N <= 0 || K <= 0 || K % 256 != 0 || N > INT32_MAX / 2 || K > (1 << 24))
    return FP4_ERR_INVALID_ARG;
  if (!aligned(w, 16) || !aligned(scales, 16)) return FP4_ERR_ALIGNMENT;
  const DevInfo* d = nullptr;
  fp4_status st = current(&d);
  if (st != FP4_OK) return st;
  if (!qmv_tc_supported(*d, FP4_MODE_NVFP4, N, K)) return FP4_ERR_UNSUPPORTED;  // no tensor-core plan
  return from_cuda(launch_weight_stream(*d, w, scales, N, K, stream));
}

fp4_status fp4_debug_inject_wait_timeout(int enable) {
  g_inject_timeout.store(enable ? 1 : 0);
  return FP4_OK;
}

}  // extern "C"
