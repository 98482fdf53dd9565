// qlin_internal.h -- host-side declarations shared by the translation units
// of libqlin (launchers called from the C ABI in qlin_api.cu).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace qlin {

// Per-device facts cached by the API layer.
struct DeviceInfo {
  int device = -1;
  int sm_count = 0;
  bool supported = false;  // sm_103
  int* err_word = nullptr; // device address of the error word
};

// Returns the cached info of the current device (nullptr if no device).
const DeviceInfo* current_device();

// The act-quant producers write the codes q as int8, or (c16) as the same
// integers in fp16 [M, K].
cudaError_t launch_act_quant(const uint16_t* x, int64_t M, int64_t K, void* q, bool c16,
                             float* s, cudaStream_t stream);

cudaError_t launch_rmsnorm_quant(const uint16_t* x, const uint16_t* gamma, float eps, int64_t M,
                                 int64_t K, void* q, bool c16, float* s, uint16_t* y, int* err,
                                 int sm_count, cudaStream_t stream);

cudaError_t launch_silu_mul_quant(const uint16_t* gate_up, int64_t M, int64_t I, void* q,
                                  bool c16, float* s, uint16_t* y, int* err, int sm_count,
                                  cudaStream_t stream);

cudaError_t launch_pack(const int8_t* q, int64_t K, int64_t N, int bits, int32_t* qweight,
                        int32_t* qzeros, int* err, cudaStream_t stream);

cudaError_t launch_wait_timeout(int64_t limit_ns, int* err, cudaStream_t stream);

cudaError_t launch_ingest_nk(const int32_t* packed_nk, const uint16_t* scales_ng, int64_t K,
                             int64_t N, int bits, int32_t* qweight, uint16_t* scales,
                             cudaStream_t stream);

// Bytes of the tile layout of a [K*bits/32, N] GPTQ weight matrix, and the
// repack into it (see tiles_kernel in pack.cu).
size_t tiles_bytes(int64_t K, int64_t N, int bits);
cudaError_t launch_pack_tiles(const int32_t* qweight, int64_t K, int64_t N, int bits,
                              int32_t* tiles, cudaStream_t stream);

// GEMM problem description passed from the API to the launcher.
enum class GemmMode : int { kW8A8 = 0, kW8A8Partials = 1, kW4A16 = 2, kW8A16 = 3 };

struct GemmArgs {
  GemmMode mode;
  const void* act;        // int8 q_a [M,K] (W8A8) or bf16 x [M,K] (W4A16)
  const float* s_a;       // W8A8 only
  const int32_t* qweight; // [K/4,N] or [K/8,N]
  const uint16_t* scales; // fp16 (W8A8) or bf16 (W4A16) [K/128,N]
  void* out;              // bf16 y [M,N] or int32 P [K/128,M,N]
  int64_t M, N, K;
  void* workspace;
  size_t workspace_bytes;
  // Greedy-argmax variant: instead of writing y, reduce every output row to
  // a 64-bit key (order-preserving bf16 bits << 32 | ~n) with atomicMax; the
  // largest key is the largest value, lowest n on ties.  nullptr = write y.
  unsigned long long* amax_keys = nullptr;
  // W8A16: K-width of a scale group (32 or 128), or 0 for one scale per column
  int group_size = 128;
  // Weights in the tile layout (qweight is then unused), else nullptr.
  const int32_t* wtiles = nullptr;
  // W8A8: act holds the codes as fp16 [M,K] (integers in [-127, 127])
  // instead of int8.
  bool act_c16 = false;
};

// Offset of the argmax keys (one per row, M <= 96) inside the fixed counter
// region at the start of the workspace.
constexpr size_t kArgmaxKeysOffset = 4096;
constexpr int64_t kArgmaxMaxRows = 96;

// idx[m] = the column index encoded in keys[m] (-1 if no key).  Programmatic
// dependent launch: waits for the GEMM that produced the keys.
cudaError_t launch_argmax_finalize(const unsigned long long* keys, int64_t M, int32_t* idx,
                                   cudaStream_t stream);

// Tiling plan for one GEMM call.
struct GemmPlan {
  int T;           // token tile (MMA N): 16, 32, 64 or 96
  int64_t F;       // feature tiles of 128
  int64_t TT;      // token tiles
  int64_t G;       // groups of 128 along K
  int64_t steps;   // TT * F * G
  int64_t ctas;    // grid size
  int64_t band;    // banded whole-tile schedule: token tiles per band (0: stream-K)
  size_t counter_bytes;
  size_t act_offset;     // W8A8 activations in the other code width: the fp16
                         // image of int8 codes (token tiles >= 64) or the int8
                         // codes of fp16 ones (token tiles <= 32)
  size_t workspace_bytes;
};

GemmPlan plan_gemm(int64_t M, int64_t N, int64_t K, int sm_count);

cudaError_t launch_gemm(const GemmArgs& a, const GemmPlan& p, int* err, cudaStream_t stream);

// Launches `kernel` with programmatic stream serialization: it may start
// before the previous kernel on the stream has finished, and must call
// griddepcontrol.wait before it touches memory that kernel produces or uses.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace qlin
