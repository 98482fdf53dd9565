// qlin_api.cu -- the extern "C" entry points of libqlin (include/qlin.h):
// argument checks, per-device state (SM count, architecture, the device error
// word) and dispatch to the launchers.  No call allocates device memory.
#include <cmath>
#include <mutex>

#include "../../include/qlin.h"
#include "qlin_device.cuh"
#include "qlin_internal.h"

namespace qlin {

// Device-wide error word: [0] = code, [1] = where, [2] = block, [3] = spare.
__device__ int g_error_word[4];

namespace {

constexpr int kMaxDevices = 64;
DeviceInfo g_devices[kMaxDevices];
std::once_flag g_device_once[kMaxDevices];

void init_device(int dev) {
  DeviceInfo& d = g_devices[dev];
  d.device = dev;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return;
  }
  d.supported = (major == 10 && minor == 3);
  if (!d.supported) return;
  void* addr = nullptr;
  if (cudaGetSymbolAddress(&addr, g_error_word) != cudaSuccess) {
    cudaGetLastError();
    d.supported = false;
    return;
  }
  d.err_word = static_cast<int*>(addr);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int64_t kMaxDim = 2147483647LL;

qlin_status_t check_gemm_shape(int64_t M, int64_t N, int64_t K) {
  if (M < 0 || M > kMaxDim || N < 8 || N > kMaxDim || (N % 8) != 0 || K < kGroup ||
      K > kMaxDim || (K % kGroup) != 0)
    return QLIN_ERR_SHAPE;
  return QLIN_OK;
}

}  // namespace

const DeviceInfo* current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return nullptr;
  }
  std::call_once(g_device_once[dev], init_device, dev);
  return &g_devices[dev];
}

}  // namespace qlin

using namespace qlin;

namespace {

qlin_status_t device_or_error(const DeviceInfo** out) {
  const DeviceInfo* d = current_device();
  if (d == nullptr || !d->supported) return QLIN_ERR_DEVICE;
  *out = d;
  return QLIN_OK;
}

qlin_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? QLIN_OK : QLIN_ERR_CUDA; }

qlin_status_t run_gemm(GemmMode mode, const void* act, const float* s_a, const int32_t* qweight,
                       const uint16_t* scales, void* out, int64_t M, int64_t N, int64_t K,
                       void* workspace, size_t workspace_bytes, cudaStream_t stream,
                       int group_size = 128, bool tiled = false, bool act_c16 = false) {
  // an empty batch reads and writes nothing: its activation, scale and
  // output pointers may be NULL.  `tiled`: qweight holds the tile layout.
  const bool rows = M != 0;
  if ((rows && (act == nullptr || out == nullptr || (mode == GemmMode::kW8A8 && s_a == nullptr))) ||
      qweight == nullptr || (mode != GemmMode::kW8A8Partials && scales == nullptr))
    return QLIN_ERR_NULL;
  qlin_status_t st = check_gemm_shape(M, N, K);
  if (st != QLIN_OK) return st;
  if (!aligned16(act) || !aligned16(qweight) || !aligned16(out) ||
      (scales && !aligned16(scales)) || (s_a && !aligned16(s_a)) ||
      (workspace && !aligned16(workspace)))
    return QLIN_ERR_ALIGN;
  const DeviceInfo* d = nullptr;
  st = device_or_error(&d);
  if (st != QLIN_OK) return st;
  if (M == 0) return QLIN_OK;
  const GemmPlan plan = plan_gemm(M, N, K, d->sm_count);
  if (workspace == nullptr || workspace_bytes < plan.workspace_bytes) return QLIN_ERR_WORKSPACE;
  GemmArgs a{mode, act, s_a, qweight, scales, out, M, N, K, workspace, workspace_bytes};
  a.group_size = group_size;
  if (tiled) a.wtiles = qweight;
  a.act_c16 = act_c16;
  return from_cuda(launch_gemm(a, plan, d->err_word, stream));
}

// Greedy-argmax variant of the two GEMMs: the keys live at a fixed offset in
// the workspace's counter region; cleared, reduced by the GEMM, decoded.
qlin_status_t run_argmax(GemmMode mode, const void* act, const float* s_a, const int32_t* qweight,
                         const uint16_t* scales, int32_t* idx, int64_t M, int64_t N, int64_t K,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  const bool rows = M != 0;
  if ((rows && (act == nullptr || idx == nullptr || (mode == GemmMode::kW8A8 && s_a == nullptr))) ||
      qweight == nullptr || scales == nullptr)
    return QLIN_ERR_NULL;
  qlin_status_t st = check_gemm_shape(M, N, K);
  if (st != QLIN_OK) return st;
  if (M > kArgmaxMaxRows) return QLIN_ERR_SHAPE;
  if (!aligned16(act) || !aligned16(qweight) || !aligned16(scales) ||
      (s_a && !aligned16(s_a)) || (workspace && !aligned16(workspace)) ||
      (reinterpret_cast<uintptr_t>(idx) & 3u) != 0)
    return QLIN_ERR_ALIGN;
  const DeviceInfo* d = nullptr;
  st = device_or_error(&d);
  if (st != QLIN_OK) return st;
  if (M == 0) return QLIN_OK;
  const GemmPlan plan = plan_gemm(M, N, K, d->sm_count);
  if (workspace == nullptr || workspace_bytes < plan.workspace_bytes) return QLIN_ERR_WORKSPACE;
  auto* keys = reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(workspace) +
                                                     kArgmaxKeysOffset);
  if (cudaMemsetAsync(keys, 0, static_cast<size_t>(M) * sizeof(unsigned long long), stream) !=
      cudaSuccess)
    return QLIN_ERR_CUDA;
  GemmArgs a{mode, act, s_a, qweight, scales, nullptr, M, N, K, workspace, workspace_bytes};
  a.amax_keys = keys;
  st = from_cuda(launch_gemm(a, plan, d->err_word, stream));
  if (st != QLIN_OK) return st;
  return from_cuda(launch_argmax_finalize(keys, M, idx, stream));
}


qlin_status_t run_act_quant(const uint16_t* x, int64_t M, int64_t K, void* q, bool c16,
                            float* s_a, cudaStream_t stream) {
  if (M != 0 && (x == nullptr || q == nullptr || s_a == nullptr)) return QLIN_ERR_NULL;
  if (M < 0 || M > kMaxDim || K < kGroup || K > kMaxDim || (K % kGroup) != 0)
    return QLIN_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(q) || !aligned16(s_a)) return QLIN_ERR_ALIGN;
  const DeviceInfo* d = nullptr;
  qlin_status_t st = device_or_error(&d);
  if (st != QLIN_OK) return st;
  if (M == 0) return QLIN_OK;
  return from_cuda(launch_act_quant(x, M, K, q, c16, s_a, stream));
}

qlin_status_t run_rmsnorm_quant(const uint16_t* x, const uint16_t* gamma, float eps, int64_t M,
                                int64_t K, void* q, bool c16, float* s_a, uint16_t* y,
                                cudaStream_t stream) {
  if (gamma == nullptr || (M != 0 && (x == nullptr || q == nullptr || s_a == nullptr)))
    return QLIN_ERR_NULL;
  if (M < 0 || M > kMaxDim || K < kGroup || K > kMaxDim || (K % kGroup) != 0 || !(eps >= 0.0f) ||
      !std::isfinite(eps))
    return QLIN_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(gamma) || !aligned16(q) || !aligned16(s_a) ||
      (y != nullptr && !aligned16(y)))
    return QLIN_ERR_ALIGN;
  const DeviceInfo* d = nullptr;
  qlin_status_t st = device_or_error(&d);
  if (st != QLIN_OK) return st;
  if (M == 0) return QLIN_OK;
  return from_cuda(
      launch_rmsnorm_quant(x, gamma, eps, M, K, q, c16, s_a, y, d->err_word, d->sm_count, stream));
}

qlin_status_t run_silu_mul_quant(const uint16_t* gate_up, int64_t M, int64_t I, void* q, bool c16,
                                 float* s_a, uint16_t* y, cudaStream_t stream) {
  if (M != 0 && (gate_up == nullptr || q == nullptr || s_a == nullptr)) return QLIN_ERR_NULL;
  if (M < 0 || M > kMaxDim || I < kGroup || I > kMaxDim || (I % kGroup) != 0)
    return QLIN_ERR_SHAPE;
  if (!aligned16(gate_up) || !aligned16(q) || !aligned16(s_a) || (y != nullptr && !aligned16(y)))
    return QLIN_ERR_ALIGN;
  const DeviceInfo* d = nullptr;
  qlin_status_t st = device_or_error(&d);
  if (st != QLIN_OK) return st;
  if (M == 0) return QLIN_OK;
  return from_cuda(
      launch_silu_mul_quant(gate_up, M, I, q, c16, s_a, y, d->err_word, d->sm_count, stream));
}

}  // namespace

extern "C" {

qlin_status_t qlin_act_quant_i8(const uint16_t* x, int64_t M, int64_t K, int8_t* q, float* s_a,
                                qlin_stream_t stream) {
  return run_act_quant(x, M, K, q, false, s_a, reinterpret_cast<cudaStream_t>(stream));
}

qlin_status_t qlin_act_quant_c16(const uint16_t* x, int64_t M, int64_t K, uint16_t* q,
                                 float* s_a, qlin_stream_t stream) {
  return run_act_quant(x, M, K, q, true, s_a, reinterpret_cast<cudaStream_t>(stream));
}

qlin_status_t qlin_rmsnorm_act_quant_i8(const uint16_t* x, const uint16_t* gamma, float eps,
                                        int64_t M, int64_t K, int8_t* q, float* s_a, uint16_t* y,
                                        qlin_stream_t stream) {
  return run_rmsnorm_quant(x, gamma, eps, M, K, q, false, s_a, y,
                           reinterpret_cast<cudaStream_t>(stream));
}

qlin_status_t qlin_rmsnorm_act_quant_c16(const uint16_t* x, const uint16_t* gamma, float eps,
                                         int64_t M, int64_t K, uint16_t* q, float* s_a,
                                         uint16_t* y, qlin_stream_t stream) {
  return run_rmsnorm_quant(x, gamma, eps, M, K, q, true, s_a, y,
                           reinterpret_cast<cudaStream_t>(stream));
}

qlin_status_t qlin_silu_mul_act_quant_i8(const uint16_t* gate_up, int64_t M, int64_t I, int8_t* q,
                                         float* s_a, uint16_t* y, qlin_stream_t stream) {
  return run_silu_mul_quant(gate_up, M, I, q, false, s_a, y,
                            reinterpret_cast<cudaStream_t>(stream));
}

qlin_status_t qlin_silu_mul_act_quant_c16(const uint16_t* gate_up, int64_t M, int64_t I,
                                          uint16_t* q, float* s_a, uint16_t* y,
                                          qlin_stream_t stream) {
  return run_silu_mul_quant(gate_up, M, I, q, true, s_a, y,
                            reinterpret_cast<cudaStream_t>(stream));
}

qlin_status_t qlin_gemm_w8a8_gs128(const int8_t* q_a, const float* s_a, const int32_t* qweight,
                                   const uint16_t* scales, int64_t M, int64_t N, int64_t K,
                                   uint16_t* y, void* workspace, size_t workspace_bytes,
                                   qlin_stream_t stream) {
  return run_gemm(GemmMode::kW8A8, q_a, s_a, qweight, scales, y, M, N, K, workspace,
                  workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

qlin_status_t qlin_gemm_w8a8_gs128_c16(const uint16_t* q_a, const float* s_a,
                                       const int32_t* qweight, const uint16_t* scales, int64_t M,
                                       int64_t N, int64_t K, uint16_t* y, void* workspace,
                                       size_t workspace_bytes, qlin_stream_t stream) {
  return run_gemm(GemmMode::kW8A8, q_a, s_a, qweight, scales, y, M, N, K, workspace,
                  workspace_bytes, reinterpret_cast<cudaStream_t>(stream), 128, false, true);
}

qlin_status_t qlin_gemm_w8a8_gs128_tiled(const int8_t* q_a, const float* s_a, const int32_t* tiles,
                                         const uint16_t* scales, int64_t M, int64_t N, int64_t K,
                                         uint16_t* y, void* workspace, size_t workspace_bytes,
                                         qlin_stream_t stream) {
  return run_gemm(GemmMode::kW8A8, q_a, s_a, tiles, scales, y, M, N, K, workspace,
                  workspace_bytes, reinterpret_cast<cudaStream_t>(stream), 128, true);
}

qlin_status_t qlin_gemm_w4a16_g128_tiled(const uint16_t* x, const int32_t* tiles,
                                         const uint16_t* scales, int64_t M, int64_t N, int64_t K,
                                         uint16_t* y, void* workspace, size_t workspace_bytes,
                                         qlin_stream_t stream) {
  return run_gemm(GemmMode::kW4A16, x, nullptr, tiles, scales, y, M, N, K, workspace,
                  workspace_bytes, reinterpret_cast<cudaStream_t>(stream), 128, true);
}

qlin_status_t qlin_gemm_w4a16_g128(const uint16_t* x, const int32_t* qweight,
                                   const uint16_t* scales, int64_t M, int64_t N, int64_t K,
                                   uint16_t* y, void* workspace, size_t workspace_bytes,
                                   qlin_stream_t stream) {
  return run_gemm(GemmMode::kW4A16, x, nullptr, qweight, scales, y, M, N, K, workspace,
                  workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

qlin_status_t qlin_gemm_w8a16(const uint16_t* x, const int32_t* qweight, const uint16_t* scales,
                              int64_t M, int64_t N, int64_t K, int group_size, uint16_t* y,
                              void* workspace, size_t workspace_bytes, qlin_stream_t stream) {
  if (group_size != 0 && group_size != 32 && group_size != 128) return QLIN_ERR_SHAPE;
  return run_gemm(GemmMode::kW8A16, x, nullptr, qweight, scales, y, M, N, K, workspace,
                  workspace_bytes, reinterpret_cast<cudaStream_t>(stream), group_size);
}

qlin_status_t qlin_gemm_w8a8_gs128_argmax(const int8_t* q_a, const float* s_a,
                                          const int32_t* qweight, const uint16_t* scales,
                                          int64_t M, int64_t N, int64_t K, int32_t* argmax,
                                          void* workspace, size_t workspace_bytes,
                                          qlin_stream_t stream) {
  return run_argmax(GemmMode::kW8A8, q_a, s_a, qweight, scales, argmax, M, N, K, workspace,
                    workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

qlin_status_t qlin_gemm_w4a16_g128_argmax(const uint16_t* x, const int32_t* qweight,
                                          const uint16_t* scales, int64_t M, int64_t N, int64_t K,
                                          int32_t* argmax, void* workspace,
                                          size_t workspace_bytes, qlin_stream_t stream) {
  return run_argmax(GemmMode::kW4A16, x, nullptr, qweight, scales, argmax, M, N, K, workspace,
                    workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

qlin_status_t qlin_debug_group_partials_i8(const int8_t* q_a, const int32_t* qweight, int64_t M,
                                           int64_t N, int64_t K, int32_t* P, void* workspace,
                                           size_t workspace_bytes, qlin_stream_t stream) {
  return run_gemm(GemmMode::kW8A8Partials, q_a, nullptr, qweight, nullptr, P, M, N, K, workspace,
                  workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

qlin_status_t qlin_ingest_nk(const int32_t* packed_nk, const uint16_t* scales_ng, int64_t K,
                             int64_t N, int bits, int32_t* qweight, uint16_t* scales,
                             qlin_stream_t stream) {
  if (packed_nk == nullptr || scales_ng == nullptr || qweight == nullptr || scales == nullptr)
    return QLIN_ERR_NULL;
  if (bits != 4 && bits != 8) return QLIN_ERR_BITS;
  if (N < 1 || N > kMaxDim || K < kGroup || K > kMaxDim || (K % kGroup) != 0)
    return QLIN_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(packed_nk) & 3u) || (reinterpret_cast<uintptr_t>(scales_ng) & 1u) ||
      !aligned16(qweight) || !aligned16(scales))
    return QLIN_ERR_ALIGN;
  const DeviceInfo* d = nullptr;
  qlin_status_t st = device_or_error(&d);
  if (st != QLIN_OK) return st;
  return from_cuda(launch_ingest_nk(packed_nk, scales_ng, K, N, bits, qweight, scales,
                                    reinterpret_cast<cudaStream_t>(stream)));
}

qlin_status_t qlin_pack_gptq(const int8_t* q, int64_t K, int64_t N, int bits, int32_t* qweight,
                             int32_t* qzeros, qlin_stream_t stream) {
  if (q == nullptr || qweight == nullptr) return QLIN_ERR_NULL;
  if (bits != 4 && bits != 8) return QLIN_ERR_BITS;
  if (K < kGroup || K > kMaxDim || (K % kGroup) != 0 || N < 1 || N > kMaxDim)
    return QLIN_ERR_SHAPE;
  if (qzeros != nullptr && (N * bits) % 32 != 0) return QLIN_ERR_SHAPE;
  if (!aligned16(q) || !aligned16(qweight) || (qzeros && !aligned16(qzeros))) return QLIN_ERR_ALIGN;
  const DeviceInfo* d = nullptr;
  qlin_status_t st = device_or_error(&d);
  if (st != QLIN_OK) return st;
  return from_cuda(launch_pack(q, K, N, bits, qweight, qzeros, d->err_word,
                               reinterpret_cast<cudaStream_t>(stream)));
}

size_t qlin_tiles_bytes(int64_t K, int64_t N, int bits) {
  if ((bits != 4 && bits != 8) || N < 1 || N > kMaxDim || K < kGroup || K > kMaxDim ||
      (K % kGroup) != 0)
    return 0;
  return tiles_bytes(K, N, bits);
}

qlin_status_t qlin_pack_tiles(const int32_t* qweight, int64_t K, int64_t N, int bits,
                              int32_t* tiles, qlin_stream_t stream) {
  if (qweight == nullptr || tiles == nullptr) return QLIN_ERR_NULL;
  if (bits != 4 && bits != 8) return QLIN_ERR_BITS;
  if (N < 1 || N > kMaxDim || K < kGroup || K > kMaxDim || (K % kGroup) != 0)
    return QLIN_ERR_SHAPE;
  if (!aligned16(qweight) || !aligned16(tiles)) return QLIN_ERR_ALIGN;
  const DeviceInfo* d = nullptr;
  qlin_status_t st = device_or_error(&d);
  if (st != QLIN_OK) return st;
  return from_cuda(launch_pack_tiles(qweight, K, N, bits, tiles,
                                     reinterpret_cast<cudaStream_t>(stream)));
}

size_t qlin_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  if (check_gemm_shape(M, N, K) != QLIN_OK || M == 0) return 0;
  const DeviceInfo* d = current_device();
  if (d == nullptr || !d->supported) return 0;
  return plan_gemm(M, N, K, d->sm_count).workspace_bytes;
}

qlin_status_t qlin_debug_wait_timeout(int64_t limit_ns, qlin_stream_t stream) {
  if (limit_ns < 1000 || limit_ns > 10000000000LL) return QLIN_ERR_SHAPE;
  const DeviceInfo* d = nullptr;
  qlin_status_t st = device_or_error(&d);
  if (st != QLIN_OK) return st;
  return from_cuda(launch_wait_timeout(limit_ns, d->err_word, reinterpret_cast<cudaStream_t>(stream)));
}

qlin_status_t qlin_device_status(qlin_stream_t stream) {
  const DeviceInfo* d = nullptr;
  qlin_status_t st = device_or_error(&d);
  if (st != QLIN_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return QLIN_ERR_CUDA;
  int word[4] = {0, 0, 0, 0};
  if (cudaMemcpy(word, d->err_word, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return QLIN_ERR_CUDA;
  if (word[0] != 0) {
    const int zero[4] = {0, 0, 0, 0};
    if (cudaMemcpy(d->err_word, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
      return QLIN_ERR_CUDA;
  }
  if (word[0] == kDevTimeout) return QLIN_ERR_DEVICE_TIMEOUT;
  if (word[0] == kDevValueRange) return QLIN_ERR_VALUE_RANGE;
  return QLIN_OK;
}

qlin_status_t qlin_device_error_detail(qlin_stream_t stream, int32_t* where, int32_t* block) {
  const DeviceInfo* d = nullptr;
  qlin_status_t st = device_or_error(&d);
  if (st != QLIN_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return QLIN_ERR_CUDA;
  int word[4] = {0, 0, 0, 0};
  if (cudaMemcpy(word, d->err_word, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return QLIN_ERR_CUDA;
  if (where) *where = word[1];
  if (block) *block = word[2];
  if (word[0] == kDevTimeout) return QLIN_ERR_DEVICE_TIMEOUT;
  if (word[0] == kDevValueRange) return QLIN_ERR_VALUE_RANGE;
  return QLIN_OK;
}

const char* qlin_status_string(qlin_status_t status) {
  switch (status) {
    case QLIN_OK: return "ok";
    case QLIN_ERR_NULL: return "a required pointer is NULL";
    case QLIN_ERR_SHAPE: return "invalid shape (K must be a positive multiple of 128, N a positive multiple of 8)";
    case QLIN_ERR_ALIGN: return "a pointer is not 16-byte aligned";
    case QLIN_ERR_WORKSPACE: return "workspace is NULL or smaller than qlin_workspace_bytes()";
    case QLIN_ERR_BITS: return "bits must be 4 or 8";
    case QLIN_ERR_DEVICE: return "the current device is not an sm_103 GPU";
    case QLIN_ERR_TOO_LARGE: return "the problem needs more scratch than the no-alloc entry's 24 MiB array";
    case QLIN_ERR_CUDA: return "a CUDA call or kernel launch failed";
    case QLIN_ERR_DEVICE_TIMEOUT: return "a bounded wait inside a kernel ran out";
    case QLIN_ERR_VALUE_RANGE: return "the packer met a value outside the bit width";
    default: return "unknown status";
  }
}

int qlin_version(void) { return 103; }

}  // extern "C"
