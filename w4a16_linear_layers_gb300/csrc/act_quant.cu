// act_quant.cu -- dynamic per-token symmetric INT8 activation quantization.
//
// Passages: "Flint-DFlash2-GPTQ-INT8-PTQR" model card (dynamic per-token
// activation quantization; VLLM_GFX908_ACT_QUANT=round) and
// "Qwen3.8-27B-GPTQ-INT8-W8A8-GS128-PTQR" card, "Serving" (GEMM inputs are
// dynamically quantized to INT8).
//
// One block of 256 threads per row.  The row is read once with 16-byte
// vector loads and kept in registers (rows of up to 32768 elements; longer
// rows are read twice, the second time from L2); the row maximum of |x| is
// reduced with warp shuffles and one shared-memory step; then
// s = amax / 127 and q = rint(x / s) are formed with IEEE fp32 division
// (div.rn), exactly as the format defines them, and written as 8-byte stores.
#include <cuda_bf16.h>

#include "qlin_device.cuh"
#include "qlin_internal.h"

namespace qlin {
namespace {

constexpr int kAqThreads = 256;
constexpr int kAqVecPerThread = 16;  // 16 x 8 bf16 = 128 elements per thread in registers

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float absmax8(uint4 v, float m) {
  m = fmaxf(m, fabsf(bf16_lo(v.x)));
  m = fmaxf(m, fabsf(bf16_hi(v.x)));
  m = fmaxf(m, fabsf(bf16_lo(v.y)));
  m = fmaxf(m, fabsf(bf16_hi(v.y)));
  m = fmaxf(m, fabsf(bf16_lo(v.z)));
  m = fmaxf(m, fabsf(bf16_hi(v.z)));
  m = fmaxf(m, fabsf(bf16_lo(v.w)));
  m = fmaxf(m, fabsf(bf16_hi(v.w)));
  return m;
}

__device__ __forceinline__ uint32_t quant1(float x, float s) {
  // IEEE division (no fast-math in this build), round half to even, clamp.
  float r = rintf(__fdiv_rn(x, s));
  r = fminf(fmaxf(r, -127.0f), 127.0f);
  return static_cast<uint32_t>(static_cast<int>(r)) & 0xFFu;
}

__device__ __forceinline__ uint2 quant8(uint4 v, float s) {
  uint2 o;
  o.x = quant1(bf16_lo(v.x), s) | (quant1(bf16_hi(v.x), s) << 8) |
        (quant1(bf16_lo(v.y), s) << 16) | (quant1(bf16_hi(v.y), s) << 24);
  o.y = quant1(bf16_lo(v.z), s) | (quant1(bf16_hi(v.z), s) << 8) |
        (quant1(bf16_lo(v.w), s) << 16) | (quant1(bf16_hi(v.w), s) << 24);
  return o;
}

template <bool kCached>
__global__ void __launch_bounds__(kAqThreads) act_quant_kernel(const uint16_t* __restrict__ x,
                                                               int64_t K, int8_t* __restrict__ q,
                                                               float* __restrict__ s_out) {
  __shared__ float red[kAqThreads / 32];
  // Launched with programmatic serialization: wait for the previous kernel
  // (which may produce x or still read q) before touching memory, then let
  // the next kernel (a GEMM that streams weights first) start.
  grid_dep_wait();
  grid_dep_launch();
  const int64_t m = blockIdx.x;
  const int64_t nvec = K / 8;
  const uint4* row = reinterpret_cast<const uint4*>(x + m * K);
  uint2* qrow = reinterpret_cast<uint2*>(q + m * K);
  const int tid = threadIdx.x;

  uint4 cache[kCached ? kAqVecPerThread : 1];
  float amax = 0.0f;
  if (kCached) {
#pragma unroll
    for (int i = 0; i < kAqVecPerThread; ++i) {
      const int64_t v = tid + static_cast<int64_t>(i) * kAqThreads;
      if (v < nvec) {
        cache[i] = __ldg(row + v);
        amax = absmax8(cache[i], amax);
      }
    }
  } else {
    for (int64_t v = tid; v < nvec; v += kAqThreads) amax = absmax8(__ldg(row + v), amax);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
  if ((tid & 31) == 0) red[tid >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int w = 1; w < kAqThreads / 32; ++w) amax = fmaxf(amax, red[w]);

  const float s = __fdiv_rn(amax, 127.0f);
  if (tid == 0) s_out[m] = s;
  if (amax == 0.0f) {
    for (int64_t v = tid; v < nvec; v += kAqThreads) qrow[v] = make_uint2(0u, 0u);
    return;
  }
  if (kCached) {
#pragma unroll
    for (int i = 0; i < kAqVecPerThread; ++i) {
      const int64_t v = tid + static_cast<int64_t>(i) * kAqThreads;
      if (v < nvec) qrow[v] = quant8(cache[i], s);
    }
  } else {
    for (int64_t v = tid; v < nvec; v += kAqThreads) qrow[v] = quant8(__ldg(row + v), s);
  }
}

}  // namespace

cudaError_t launch_act_quant(const uint16_t* x, int64_t M, int64_t K, int8_t* q, float* s,
                             cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>(M));
  if (K <= static_cast<int64_t>(kAqThreads) * kAqVecPerThread * 8)
    return launch_pdl(act_quant_kernel<true>, grid, dim3(kAqThreads), 0, stream, x, K, q, s);
  return launch_pdl(act_quant_kernel<false>, grid, dim3(kAqThreads), 0, stream, x, K, q, s);
}

}  // namespace qlin
