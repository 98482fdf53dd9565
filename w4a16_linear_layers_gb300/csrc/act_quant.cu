// act_quant.cu -- dynamic per-token symmetric INT8 activation quantization,
// alone and fused into the producers of the projections' inputs.
//
// Passages: "Flint-DFlash2-GPTQ-INT8-PTQR" model card (dynamic per-token
// activation quantization; VLLM_GFX908_ACT_QUANT=round);
// "Qwen3.8-27B-GPTQ-INT8-W8A8-GS128-PTQR" card, "Serving" (GEMM inputs are
// dynamically quantized to INT8); "Qwen3.8-27B-DFlash2-W4A16-g128-sym-GPTQ"
// card (the BF16 norms in front of the q/k/v and gate/up projections, the
// gated MLP in front of down_proj).
//
// act_quant_kernel: one block per row (1024 threads for up to 256 rows, else
// 256).  The row is read once with 16-byte vector loads and kept in registers
// (rows of up to 32768 elements; longer rows are read twice, the second time
// from L2).  The row maximum of |x| is reduced with warp shuffles and one
// shared-memory step; s = amax / 127 is an IEEE fp32 divide, and the codes are
// those of rint(x / s) with an IEEE divide (quant1y), written as 8-byte
// stores of int8, or for the _c16 calls as the same integers in fp16 (16-byte
// stores), the W8A8 GEMM's tensor-core operand type.  The producer kernels
// are described at "fused producers" below.
#include <cuda_bf16.h>

#include <mutex>

#include "qlin_device.cuh"
#include "qlin_internal.h"

namespace qlin {
namespace {

constexpr int kAqThreads = 256;        // the long-row producer kernels
constexpr int kAqRowVecs = 4096;       // rows of up to 4096 x 8 elements stay in registers

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

// The same code from the reciprocal y = 1/s (correctly rounded) instead of a
// divide per element.  t = x * y is within 2^-16 of x / s for |x / s| <= 127,
// so when t is further than 2^-15 from a half-integer, the IEEE quotient
// rounds to the same integer as t; the rare values near a rounding boundary
// take the IEEE divide.  The codes are those of quant1 in every case.
__device__ __forceinline__ uint32_t quant1y(float x, float s, float y) {
  const float t = __fmul_rn(x, y);
  float r = rintf(t);
  if (fabsf(__fsub_rn(t, r)) > 0.5f - 0x1p-15f) r = rintf(__fdiv_rn(x, s));
  r = fminf(fmaxf(r, -127.0f), 127.0f);
  return static_cast<uint32_t>(static_cast<int>(r)) & 0xFFu;
}

__device__ __forceinline__ uint2 quant8y(uint4 v, float s, float y) {
  uint2 o;
  o.x = quant1y(bf16_lo(v.x), s, y) | (quant1y(bf16_hi(v.x), s, y) << 8) |
        (quant1y(bf16_lo(v.y), s, y) << 16) | (quant1y(bf16_hi(v.y), s, y) << 24);
  o.y = quant1y(bf16_lo(v.z), s, y) | (quant1y(bf16_hi(v.z), s, y) << 8) |
        (quant1y(bf16_lo(v.w), s, y) << 16) | (quant1y(bf16_hi(v.w), s, y) << 24);
  return o;
}

// The codes of one row: int8, or (c16) the same integers as fp16 values,
// which the W8A8 GEMM's tensor cores read without a conversion pass.
// Each store takes 8 consecutive codes (element 8v .. 8v + 7 of the row).
struct CodeRow {
  void* base;
  bool c16;
  __device__ __forceinline__ CodeRow(void* q, int64_t row_elems, int64_t m, bool c16_)
      : base(c16_ ? static_cast<void*>(static_cast<uint16_t*>(q) + m * row_elems)
                  : static_cast<void*>(static_cast<int8_t*>(q) + m * row_elems)),
        c16(c16_) {}
  __device__ __forceinline__ void store(int64_t v, uint2 codes) const {
    if (!c16) {
      reinterpret_cast<uint2*>(base)[v] = codes;
    } else {
      uint4 o;
      biased_u8x4_to_f16x4(codes.x ^ 0x80808080u, o.x, o.y);
      biased_u8x4_to_f16x4(codes.y ^ 0x80808080u, o.z, o.w);
      reinterpret_cast<uint4*>(base)[v] = o;
    }
  }
};

// kThreads threads per row: 1024 for small batches (each row's latency is the
// whole call's), 256 for many rows (several blocks per SM).
template <bool kCached, int kThreads>
__global__ void __launch_bounds__(kThreads) act_quant_kernel(const uint16_t* __restrict__ x,
                                                             int64_t K, void* __restrict__ q,
                                                             float* __restrict__ s_out, bool c16) {
  constexpr int kVec = kAqRowVecs / kThreads;
  __shared__ float red[kThreads / 32];
  // Launched with programmatic serialization: wait for the previous kernel
  // (which may produce x or still read q) before touching memory, then let
  // the next kernel (a GEMM that streams weights first) start.
  grid_dep_wait();
  grid_dep_launch();
  const int64_t m = blockIdx.x;
  const int64_t nvec = K / 8;
  const uint4* row = reinterpret_cast<const uint4*>(x + m * K);
  const CodeRow qrow(q, K, m, c16);
  const int tid = threadIdx.x;

  uint4 cache[kCached ? kVec : 1];
  float amax = 0.0f;
  if (kCached) {
#pragma unroll
    for (int i = 0; i < kVec; ++i) {
      const int64_t v = tid + static_cast<int64_t>(i) * kThreads;
      if (v < nvec) {
        cache[i] = __ldg(row + v);
        amax = absmax8(cache[i], amax);
      }
    }
  } else {
    for (int64_t v = tid; v < nvec; v += kThreads) amax = absmax8(__ldg(row + v), amax);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
  if ((tid & 31) == 0) red[tid >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int w = 1; w < kThreads / 32; ++w) amax = fmaxf(amax, red[w]);

  const float s = __fdiv_rn(amax, 127.0f);
  if (tid == 0) s_out[m] = s;
  if (amax == 0.0f) {
    for (int64_t v = tid; v < nvec; v += kThreads) qrow.store(v, make_uint2(0u, 0u));
    return;
  }
  const float y = __frcp_rn(s);
  if (kCached) {
#pragma unroll
    for (int i = 0; i < kVec; ++i) {
      const int64_t v = tid + static_cast<int64_t>(i) * kThreads;
      if (v < nvec) qrow.store(v, quant8y(cache[i], s, y));
    }
  } else {
    for (int64_t v = tid; v < nvec; v += kThreads) qrow.store(v, quant8y(__ldg(row + v), s, y));
  }
}

// ------------------------------------------------------ fused producers
//
// The kernels that produce a linear's input, fused with its act-quant: one
// read of the producer's input and one write of q and s_a, instead of a bf16
// round trip through memory between the producer and act-quant.  The
// producer's bf16 output z is formed exactly as the unfused producer would
// store it, and quantized exactly as act_quant_kernel does; it is also
// written out when y is not null.

__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float t = red[0];
#pragma unroll
  for (int w = 1; w < kAqThreads / 32; ++w) t = fmaxf(t, red[w]);
  return t;
}

// ---- exact producer outputs
//
// The producers' bf16 outputs are the oracle's: each value is first formed in
// fp32, and where that fp32 value lies so close to a point halfway between
// two bf16 values that its known error could put the exact value on the other
// side, the value is formed again in fp64 and rounded from there.

// v added into the unevaluated sum s + c without rounding error in the
// transformation (Knuth's TwoSum); c collects what each addition dropped.
__device__ __forceinline__ void df_add(float& s, float& c, float v) {
  const float t = __fadd_rn(s, v);
  const float bp = __fsub_rn(t, s);
  const float ap = __fsub_rn(t, bp);
  c = __fadd_rn(c, __fadd_rn(__fsub_rn(s, ap), __fsub_rn(v, bp)));
  s = t;
}

// Squares of 8 bf16 values (each exact in fp32: 8 significant bits squared)
// added into s + c.
__device__ __forceinline__ void sumsq8(uint4 v, float& s, float& c) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    df_add(s, c, __fmul_rn(bf16_lo(w[i]), bf16_lo(w[i])));
    df_add(s, c, __fmul_rn(bf16_hi(w[i]), bf16_hi(w[i])));
  }
}

// True when the fp32 value with bits u is within k fp32 ulps of a point
// halfway between two bf16 values (low 16 bits 0x8000), in either direction.
__device__ __forceinline__ bool near_bf16_half(uint32_t u, uint32_t k) {
  return ((u & 0xFFFFu) - (0x8000u - k)) <= 2u * k;
}

__device__ __forceinline__ uint32_t bf16_bits_rn(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// bf16 bits of a binary64 value rounded once to nearest even: through the
// nearest fp32 value f, which rounds to the same bf16 value unless f is
// itself a halfway point; then the fp64 value picks the side.
__device__ __forceinline__ uint32_t f64_to_bf16_bits(double d) {
  const float f = __double2float_rn(d);
  const uint32_t u = __float_as_uint(f);
  if ((u & 0xFFFFu) == 0x8000u) {
    const double back = static_cast<double>(f);
    if (d != back) return fabs(d) > fabs(back) ? ((u >> 16) + 1u) & 0xFFFFu : (u >> 16);
  }
  return bf16_bits_rn(f);
}

// The norm's scale 1 / sqrt(ss / K + eps), formed once per row in fp64 from
// the compensated sum of squares; rhi is its nearest fp32 value.
struct RowScale {
  double rstd;
  float rhi;
};

__device__ __forceinline__ RowScale row_scale(double ss, int64_t K, float eps) {
  const double r = 1.0 / sqrt(ss / static_cast<double>(K) + static_cast<double>(eps));
  return RowScale{r, __double2float_rn(r)};
}

// t = bf16(x * rstd).  x * rhi in fp32 is within 2 fp32 ulps of x * rstd (rhi
// and the product each rounded once), so its bf16 rounding is the exact
// one unless it lies within 4 ulps of a halfway point; those are formed in
// fp64.
__device__ __forceinline__ float norm_t(float x, const RowScale& rs) {
  const float t = __fmul_rn(x, rs.rhi);
  const uint32_t b = near_bf16_half(__float_as_uint(t), 4u)
                         ? f64_to_bf16_bits(static_cast<double>(x) * rs.rstd)
                         : bf16_bits_rn(t);
  return __uint_as_float(b << 16);
}

// RMSNorm output of 2 elements: t = bf16(x * rstd), z = bf16(gamma * t) (the
// product of two bf16 values is exact in fp32, so z is rounded once).
__device__ __forceinline__ uint32_t norm2(uint32_t x, uint32_t g, const RowScale& rs) {
  return bf16x2_rn(__fmul_rn(bf16_lo(g), norm_t(bf16_lo(x), rs)),
                   __fmul_rn(bf16_hi(g), norm_t(bf16_hi(x), rs)));
}

__device__ __forceinline__ uint4 norm8(uint4 x, uint4 g, const RowScale& rs) {
  return make_uint4(norm2(x.x, g.x, rs), norm2(x.y, g.y, rs), norm2(x.z, g.z, rs),
                    norm2(x.w, g.w, rs));
}

// bf16(SiLU(g) * u).  In fp32: SiLU(g) = g * sigmoid(g), the sigmoid from
// e = exp(-|g|) <= 1 (1 / (1 + e) for g >= 0, e / (1 + e) below), so the
// divisor stays in [1, 2] and no exponential overflows.  With expf within 2
// ulps and the approximate divide within 2 ulps on that range (the CUDA
// programming guide's maximum-error tables), plus four roundings, the fp32
// value is within 12 ulps of the exact one; within 16 ulps of a bf16 halfway
// point it is formed again in fp64 as g / (1 + exp(-g)) * u.
// The fp64 form, out of line: it is rare (a window of 32 fp32 ulps in
// 65536), and inlined into every unrolled element it would multiply the
// kernel's code size.
__device__ __noinline__ uint32_t silu_mul_f64(float g, float u) {
  const double gd = static_cast<double>(g);
  return f64_to_bf16_bits(gd / (1.0 + exp(-gd)) * static_cast<double>(u));
}

__device__ __forceinline__ uint32_t silu_mul1(float g, float u) {
  const float e = expf(-fabsf(g));
  const float sig = __fdividef(g >= 0.0f ? 1.0f : e, __fadd_rn(1.0f, e));
  const float v = __fmul_rn(__fmul_rn(g, sig), u);
  if (near_bf16_half(__float_as_uint(v), 16u)) return silu_mul_f64(g, u);
  return bf16_bits_rn(v);
}

__device__ __forceinline__ uint32_t silu_mul2(uint32_t g, uint32_t u) {
  return silu_mul1(bf16_lo(g), bf16_lo(u)) | (silu_mul1(bf16_hi(g), bf16_hi(u)) << 16);
}

__device__ __forceinline__ uint4 silu_mul8(uint4 g, uint4 u) {
  return make_uint4(silu_mul2(g.x, u.x), silu_mul2(g.y, u.y), silu_mul2(g.z, u.z),
                    silu_mul2(g.w, u.w));
}

// Sum of the pairs (s, c) over the block, in fp64, formed by thread 0 alone
// (fp64 arithmetic is slow on this part) and returned to every thread through
// shared memory: pairs are combined across each warp with TwoSum, then
// thread 0 adds the warps' pairs in fp64.
template <int kThreads>
__device__ __forceinline__ RowScale block_row_scale(float s, float c, float2* red2,
                                                    RowScale* shared_rs, int64_t K, float eps) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float s2 = __shfl_xor_sync(0xFFFFFFFFu, s, o);
    const float c2 = __shfl_xor_sync(0xFFFFFFFFu, c, o);
    df_add(s, c, s2);
    c = __fadd_rn(c, c2);
  }
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red2[threadIdx.x >> 5] = make_float2(s, c);
  __syncthreads();
  if (threadIdx.x == 0) {
    double ss = 0.0;
#pragma unroll 1
    for (int w = 0; w < kThreads / 32; ++w)
      ss += static_cast<double>(red2[w].x) + static_cast<double>(red2[w].y);
    *shared_rs = row_scale(ss, K, eps);
  }
  __syncthreads();
  return *shared_rs;
}

// Rows longer than the persistent form holds (more than 32768 elements): one
// block per row, the row read from memory on each pass (the second and third
// from L2).  The norm: the compensated sum of squares, rstd in fp64 (once per
// row), z, then act-quant of z.
__global__ void __launch_bounds__(kAqThreads) rmsnorm_quant_long_kernel(
    const uint16_t* __restrict__ x, const uint16_t* __restrict__ gamma, float eps, int64_t K,
    void* __restrict__ q, float* __restrict__ s_out, uint16_t* __restrict__ y, bool c16) {
  __shared__ float red[kAqThreads / 32];
  __shared__ float2 red2[kAqThreads / 32];
  __shared__ RowScale row_rs;
  grid_dep_wait();
  grid_dep_launch();
  const int64_t m = blockIdx.x;
  const int64_t nvec = K / 8;
  const uint4* row = reinterpret_cast<const uint4*>(x + m * K);
  const uint4* grow = reinterpret_cast<const uint4*>(gamma);
  const CodeRow qrow(q, K, m, c16);
  uint4* yrow = y ? reinterpret_cast<uint4*>(y + m * K) : nullptr;
  const int tid = threadIdx.x;
  float ss = 0.0f, sc = 0.0f;
  for (int64_t v = tid; v < nvec; v += kAqThreads) sumsq8(__ldg(row + v), ss, sc);
  const RowScale rstd = block_row_scale<kAqThreads>(ss, sc, red2, &row_rs, K, eps);
  float amax = 0.0f;
  for (int64_t v = tid; v < nvec; v += kAqThreads) {
    const uint4 z = norm8(__ldg(row + v), __ldg(grow + v), rstd);
    amax = absmax8(z, amax);
    if (yrow) yrow[v] = z;
  }
  amax = block_max(amax, red);
  const float s = __fdiv_rn(amax, 127.0f);
  if (tid == 0) s_out[m] = s;
  for (int64_t v = tid; v < nvec; v += kAqThreads)
    qrow.store(v, amax == 0.0f ? make_uint2(0u, 0u)
                               : quant8(norm8(__ldg(row + v), __ldg(grow + v), rstd), s));
}

// The same for SiLU(gate) * up rows of more than 32768 elements.
__global__ void __launch_bounds__(kAqThreads) silu_mul_quant_long_kernel(
    const uint16_t* __restrict__ gate_up, int64_t I, void* __restrict__ q,
    float* __restrict__ s_out, uint16_t* __restrict__ y, bool c16) {
  __shared__ float red[kAqThreads / 32];
  grid_dep_wait();
  grid_dep_launch();
  const int64_t m = blockIdx.x;
  const int64_t nvec = I / 8;
  const uint4* grow = reinterpret_cast<const uint4*>(gate_up + m * 2 * I);
  const uint4* urow = grow + nvec;
  const CodeRow qrow(q, I, m, c16);
  uint4* yrow = y ? reinterpret_cast<uint4*>(y + m * I) : nullptr;
  const int tid = threadIdx.x;
  float amax = 0.0f;
  for (int64_t v = tid; v < nvec; v += kAqThreads) {
    const uint4 z = silu_mul8(__ldg(grow + v), __ldg(urow + v));
    amax = absmax8(z, amax);
    if (yrow) yrow[v] = z;
  }
  amax = block_max(amax, red);
  const float s = __fdiv_rn(amax, 127.0f);
  if (tid == 0) s_out[m] = s;
  for (int64_t v = tid; v < nvec; v += kAqThreads)
    qrow.store(v, amax == 0.0f ? make_uint2(0u, 0u)
                               : quant8(silu_mul8(__ldg(grow + v), __ldg(urow + v)), s));
}

// Persistent form for rows that fit on chip (up to 32768 elements): blocks of
// 1024 threads (rows over 8192 elements; one block per SM) or 256 threads
// (several blocks per SM) walk rows m = blockIdx.x, + gridDim.x, ...
// Each row's bf16 input lands in a shared-memory ring by one bulk copy
// (cp.async.bulk, completion on an mbarrier), issued `stages` rows ahead, so
// the next rows stream in while this one is reduced, quantized and stored.
// A ring slot is refilled as soon as every thread has copied its part of the
// row into registers (the first block-wide reduction's barrier).
constexpr int kPVec = 4;          // row vectors (8 elements) per thread
constexpr int kPMaxStages = 4;
constexpr uint32_t kPSmemBudget = 200u * 1024u;   // 1024-thread blocks
constexpr uint32_t kPSmemBudgetSmall = 44u * 1024u;   // 256-thread blocks
enum : int { kProdRms = 0, kProdSilu = 1 };

struct ProducerParams {
  const uint16_t* in;      // x [M, K] (norm) or gate_up [M, 2K] (SiLU)
  const uint16_t* gamma;   // norm weight [K]
  float eps;
  int64_t M, K;            // K: elements of one quantized row
  void* q;                 // int8 codes, or fp16 codes when c16
  float* s;
  uint16_t* y;             // optional bf16 producer output
  int* err;
  uint64_t limit_ns;
  int stages;
  uint32_t row_bytes;      // input bytes of one row
  bool c16;
};

template <int kThreads>
__device__ __forceinline__ float block_max_p(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float t = red[0];
#pragma unroll
  for (int w = 1; w < kThreads / 32; ++w) t = fmaxf(t, red[w]);
  return t;
}

template <int kKind, int kPThreads>
__global__ void __launch_bounds__(kPThreads) producer_quant_kernel(const ProducerParams p) {
  extern __shared__ uint8_t psmem_raw[];
  __shared__ uint64_t full[kPMaxStages];
  __shared__ float red[kPThreads / 32];
  __shared__ float2 red2[kPThreads / 32];
  __shared__ RowScale row_rs;
  __shared__ int abort_flag;
  uint8_t* ring = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(psmem_raw) + 127) & ~static_cast<uintptr_t>(127));
  const uint32_t ring_u32 = smem_u32(ring);
  const int tid = threadIdx.x;
  const int stages = p.stages;
  const int64_t nvec = p.K / 8;
  const int64_t in_row = kKind == kProdRms ? p.K : 2 * p.K;   // input elements per row
  const int nrows = static_cast<int>((p.M - blockIdx.x + gridDim.x - 1) / gridDim.x);
  if (tid == 0) {
    for (int i = 0; i < stages; ++i) mbar_init(smem_u32(&full[i]), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  // the input comes from the previous kernel, which may also still read q
  grid_dep_wait();
  grid_dep_launch();
  const WaitCtx ctx{p.err, &abort_flag, p.limit_ns};
  int never_abort = 0;
  const WaitCtx drain_ctx{p.err, &never_abort, p.limit_ns};
  auto issue = [&](int i) {   // thread 0: row i of this block into slot i % stages
    const int64_t m = blockIdx.x + static_cast<int64_t>(i) * gridDim.x;
    const uint32_t bar = smem_u32(&full[i % stages]);
    mbar_arrive_expect_tx(bar, p.row_bytes);
    bulk_load(ring_u32 + static_cast<uint32_t>(i % stages) * p.row_bytes, p.in + m * in_row,
              p.row_bytes, bar);
  };
  int issued = 0;
  if (tid == 0) {
    for (; issued < stages && issued < nrows; ++issued) issue(issued);
  }
  const uint4* g4 = reinterpret_cast<const uint4*>(p.gamma);
  int done = 0;
  for (int i = 0; i < nrows; ++i) {
    const int st = i % stages;
    const bool ok = mbar_wait(smem_u32(&full[st]), static_cast<uint32_t>(i / stages) & 1u, ctx, 40);
    if (!__syncthreads_and(ok)) break;
    const int64_t m = blockIdx.x + static_cast<int64_t>(i) * gridDim.x;
    const uint4* srow = reinterpret_cast<const uint4*>(ring + static_cast<uint32_t>(st) * p.row_bytes);
    uint4 z[kPVec];
    float amax = 0.0f;
    if constexpr (kKind == kProdRms) {
      float ss = 0.0f, sc = 0.0f;
#pragma unroll
      for (int j = 0; j < kPVec; ++j) {
        const int64_t v = tid + static_cast<int64_t>(j) * kPThreads;
        if (v < nvec) {
          z[j] = srow[v];
          sumsq8(z[j], ss, sc);
        }
      }
      // every thread has its part of the row in registers after the first
      // barrier of the reduction
      const RowScale rstd = block_row_scale<kPThreads>(ss, sc, red2, &row_rs, p.K, p.eps);
      if (tid == 0 && issued < nrows) {
        fence_proxy_async_smem();
        issue(issued++);
      }
#pragma unroll
      for (int j = 0; j < kPVec; ++j) {
        const int64_t v = tid + static_cast<int64_t>(j) * kPThreads;
        if (v < nvec) {
          z[j] = norm8(z[j], __ldg(g4 + v), rstd);
          amax = absmax8(z[j], amax);
        }
      }
      amax = block_max_p<kPThreads>(amax, red);
    } else {
#pragma unroll
      for (int j = 0; j < kPVec; ++j) {
        const int64_t v = tid + static_cast<int64_t>(j) * kPThreads;
        if (v < nvec) {
          z[j] = silu_mul8(srow[v], srow[nvec + v]);
          amax = absmax8(z[j], amax);
        }
      }
      amax = block_max_p<kPThreads>(amax, red);
      if (tid == 0 && issued < nrows) {
        fence_proxy_async_smem();
        issue(issued++);
      }
    }
    const float s = __fdiv_rn(amax, 127.0f);
    const float y = __frcp_rn(s);
    if (tid == 0) p.s[m] = s;
    const CodeRow qrow(p.q, p.K, m, p.c16);
    uint4* yrow = p.y ? reinterpret_cast<uint4*>(p.y + m * p.K) : nullptr;
#pragma unroll
    for (int j = 0; j < kPVec; ++j) {
      const int64_t v = tid + static_cast<int64_t>(j) * kPThreads;
      if (v < nvec) {
        qrow.store(v, amax == 0.0f ? make_uint2(0u, 0u) : quant8y(z[j], s, y));
        if (yrow) yrow[v] = z[j];
      }
    }
    done = i + 1;
  }
  // a block that gave up waits for the copies it still has in flight
  if (tid == 0) {
    for (int j = done; j < issued; ++j)
      (void)mbar_wait(smem_u32(&full[j % stages]), static_cast<uint32_t>(j / stages) & 1u, drain_ctx,
                      41);
  }
}

template <int kKind, int kThreads>
cudaError_t launch_producer_t(const ProducerParams& pp_in, int sm_count, cudaStream_t stream) {
  constexpr uint32_t budget = kThreads == 1024 ? kPSmemBudget : kPSmemBudgetSmall;
  ProducerParams pp = pp_in;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  static int per_sm = 1;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(producer_quant_kernel<kKind, kThreads>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(budget + 128));
    if (attr_err == cudaSuccess)
      attr_err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          &per_sm, producer_quant_kernel<kKind, kThreads>, kThreads, budget + 128);
    if (per_sm < 1) per_sm = 1;
  });
  if (attr_err != cudaSuccess) return attr_err;
  const int stages = static_cast<int>(budget / pp.row_bytes);
  pp.stages = stages > kPMaxStages ? kPMaxStages : stages;
  const int64_t slots = static_cast<int64_t>(sm_count) * per_sm;
  const int64_t blocks = pp.M < slots ? pp.M : slots;
  pp.limit_ns = kWaitLimitNs;
  return launch_pdl(producer_quant_kernel<kKind, kThreads>, dim3(static_cast<unsigned>(blocks)),
                    dim3(kThreads), static_cast<size_t>(pp.stages) * pp.row_bytes + 128, stream,
                    pp);
}

// Rows of up to 8192 elements take 256-thread blocks (several per SM), up to
// 32768 elements 1024-thread blocks; longer rows (or rows whose input does
// not fit the ring) return false.
template <int kKind>
bool launch_producer(const ProducerParams& pp, int sm_count, cudaStream_t stream,
                     cudaError_t* e) {
  if (pp.K <= 256 * kPVec * 8 && pp.row_bytes <= kPSmemBudgetSmall) {
    *e = launch_producer_t<kKind, 256>(pp, sm_count, stream);
    return true;
  }
  if (pp.K <= 1024 * kPVec * 8 && pp.row_bytes <= kPSmemBudget) {
    *e = launch_producer_t<kKind, 1024>(pp, sm_count, stream);
    return true;
  }
  return false;
}

}  // namespace

cudaError_t launch_rmsnorm_quant(const uint16_t* x, const uint16_t* gamma, float eps, int64_t M,
                                 int64_t K, void* q, bool c16, float* s, uint16_t* y, int* err,
                                 int sm_count, cudaStream_t stream) {
  const ProducerParams pp{x, gamma, eps, M, K, q, s, y, err, 0, 0,
                          static_cast<uint32_t>(K * 2), c16};
  cudaError_t e = cudaSuccess;
  if (K <= 32768 && launch_producer<kProdRms>(pp, sm_count, stream, &e)) return e;
  return launch_pdl(rmsnorm_quant_long_kernel, dim3(static_cast<unsigned>(M)), dim3(kAqThreads), 0,
                    stream, x, gamma, eps, K, q, s, y, c16);
}

cudaError_t launch_silu_mul_quant(const uint16_t* gate_up, int64_t M, int64_t I, void* q,
                                  bool c16, float* s, uint16_t* y, int* err, int sm_count,
                                  cudaStream_t stream) {
  const ProducerParams pp{gate_up, nullptr, 0.0f, M, I, q, s, y, err, 0, 0,
                          static_cast<uint32_t>(I * 4), c16};
  cudaError_t e = cudaSuccess;
  if (I <= 32768 && launch_producer<kProdSilu>(pp, sm_count, stream, &e)) return e;
  return launch_pdl(silu_mul_quant_long_kernel, dim3(static_cast<unsigned>(M)), dim3(kAqThreads), 0,
                    stream, gate_up, I, q, s, y, c16);
}

cudaError_t launch_act_quant(const uint16_t* x, int64_t M, int64_t K, void* q, bool c16,
                             float* s, cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>(M));
  const bool cached = K <= static_cast<int64_t>(kAqRowVecs) * 8;
  if (M <= 256)
    return cached ? launch_pdl(act_quant_kernel<true, 1024>, grid, dim3(1024), 0, stream, x, K, q,
                               s, c16)
                  : launch_pdl(act_quant_kernel<false, 1024>, grid, dim3(1024), 0, stream, x, K, q,
                               s, c16);
  return cached ? launch_pdl(act_quant_kernel<true, 256>, grid, dim3(256), 0, stream, x, K, q, s, c16)
                : launch_pdl(act_quant_kernel<false, 256>, grid, dim3(256), 0, stream, x, K, q, s,
                             c16);
}

}  // namespace qlin
