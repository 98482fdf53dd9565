// pack.cu -- GPTQ packer and the compressed-tensors ingest (offline steps),
// and the bounded-wait test kernel.
//
// Packing follows the GPTQ format of the "Flint-DFlash2-GPTQ-INT8-PTQR" card
// (qweight/qzeros, symmetric, INT8) and the INT32-packed 4-bit weights of the
// "Qwen3.8-27B-DFlash2-W4A16-g128-sym-GPTQ" card: field i of word (kk, n)
// holds q[(32/bits)*kk + i, n] + 2^(bits-1), field 0 least significant.
#include "qlin_device.cuh"
#include "qlin_internal.h"

namespace qlin {
namespace {

template <int kBits>
__global__ void pack_kernel(const int8_t* __restrict__ q, int64_t N, int64_t words,
                            int32_t* __restrict__ qweight, int* err) {
  constexpr int kPer = 32 / kBits;
  constexpr int kZero = 1 << (kBits - 1);
  constexpr uint32_t kMask = (1u << kBits) - 1u;
  bool bad = false;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < words;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t kk = i / N;
    const int64_t n = i - kk * N;
    uint32_t word = 0;
#pragma unroll
    for (int f = 0; f < kPer; ++f) {
      const int v = static_cast<int>(q[(kk * kPer + f) * N + n]) + kZero;
      bad |= (v < 0) || (v > static_cast<int>(kMask));
      word |= (static_cast<uint32_t>(v) & kMask) << (kBits * f);
    }
    qweight[i] = static_cast<int32_t>(word);
  }
  if (bad) report_error(err, kDevValueRange, 0);
}

__global__ void fill_kernel(int32_t* __restrict__ dst, int64_t count, uint32_t value) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < count;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    dst[i] = static_cast<int32_t>(value);
}

// One thread waits on a barrier that nothing completes; the bounded wait runs
// out, records kDevTimeout and the kernel returns normally.
__global__ void wait_timeout_kernel(int64_t limit_ns, int* err) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    WaitCtx ctx{err, &abort_flag, static_cast<uint64_t>(limit_ns)};
    (void)mbar_wait(smem_u32(&bar), 0, ctx, /*where=*/9999);
  }
}

// The tile layout of the GEMMs' weight stream: tile (f, g) holds the words
// of feature tile f (128 output features) and K group g (128 K values) as a
// contiguous block of W x 128 int32 (W = 32 words for 8-bit, 16 for 4-bit),
// word (kk, nl) of the tile = GPTQ word (g*W + kk, f*128 + nl); tiles are
// ordered by f, then g.  Features past N in the last tile hold 0 (never
// output).  One thread per tile word; the reads of a warp are 32 consecutive
// GPTQ words of one row and its writes 32 consecutive tile words.
__global__ void tiles_kernel(const int32_t* __restrict__ qweight, int64_t N, int64_t G, int words_per_group,
                             int64_t total, int32_t* __restrict__ tiles) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t nl = i & 127;
    const int64_t row = i >> 7;                    // (tile, kk)
    const int64_t tile = row / words_per_group;
    const int64_t kk = row - tile * words_per_group;
    const int64_t f = tile / G;
    const int64_t g = tile - f * G;
    const int64_t n = f * 128 + nl;
    tiles[i] = n < N ? qweight[(g * words_per_group + kk) * N + n] : 0;
  }
}

unsigned grid_for(int64_t n, int threads) {
  int64_t blocks = (n + threads - 1) / threads;
  if (blocks > 65535LL * 16) blocks = 65535LL * 16;
  if (blocks < 1) blocks = 1;
  return static_cast<unsigned>(blocks);
}

// dst[c][r] = src[r][c] through a 32 x 33 shared tile (both sides coalesced).
template <typename U>
__global__ void __launch_bounds__(256) transpose_kernel(const U* __restrict__ src, int64_t R,
                                                        int64_t C, U* __restrict__ dst) {
  __shared__ U tile[32][33];
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * 32;
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * 32;
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int64_t r = r0 + i, c = c0 + threadIdx.x;
    if (r < R && c < C) tile[i][threadIdx.x] = src[r * C + c];
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int64_t c = c0 + i, r = r0 + threadIdx.x;
    if (c < C && r < R) dst[c * R + r] = tile[threadIdx.x][i];
  }
}

template <typename U>
cudaError_t transpose(const U* src, int64_t R, int64_t C, U* dst, cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>((C + 31) / 32), static_cast<unsigned>((R + 31) / 32));
  transpose_kernel<U><<<grid, dim3(32, 8), 0, stream>>>(src, R, C, dst);
  return cudaGetLastError();
}

}  // namespace

// Ingest of the compressed-tensors "pack-quantized" orientation
// ("Qwen3.8-27B-DFlash2-W4A16-g128-sym-GPTQ" card, property table, Format row):
// word (n, kk) of the per-output-row packing holds the same fields as GPTQ
// word (kk, n), and the scales are [N, K/128]; the GEMMs read [K*bits/32, N]
// words and [K/128, N] scales, so both are transposed bit for bit.
cudaError_t launch_ingest_nk(const int32_t* packed_nk, const uint16_t* scales_ng, int64_t K,
                             int64_t N, int bits, int32_t* qweight, uint16_t* scales,
                             cudaStream_t stream) {
  cudaError_t e = transpose<int32_t>(packed_nk, N, K * bits / 32, qweight, stream);
  if (e != cudaSuccess) return e;
  return transpose<uint16_t>(scales_ng, N, K / kGroup, scales, stream);
}

cudaError_t launch_pack(const int8_t* q, int64_t K, int64_t N, int bits, int32_t* qweight,
                        int32_t* qzeros, int* err, cudaStream_t stream) {
  const int per = 32 / bits;
  const int64_t words = (K / per) * N;
  if (bits == 8)
    pack_kernel<8><<<grid_for(words, 256), 256, 0, stream>>>(q, N, words, qweight, err);
  else
    pack_kernel<4><<<grid_for(words, 256), 256, 0, stream>>>(q, N, words, qweight, err);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || qzeros == nullptr) return e;
  const int64_t zwords = (K / kGroup) * (N / per);
  const uint32_t zword = bits == 8 ? 0x80808080u : 0x88888888u;
  fill_kernel<<<grid_for(zwords, 256), 256, 0, stream>>>(qzeros, zwords, zword);
  return cudaGetLastError();
}

size_t tiles_bytes(int64_t K, int64_t N, int bits) {
  const int64_t F = (N + 127) / 128;
  return static_cast<size_t>(F) * static_cast<size_t>(K) * 128u * static_cast<size_t>(bits) / 8u;
}

cudaError_t launch_pack_tiles(const int32_t* qweight, int64_t K, int64_t N, int bits,
                              int32_t* tiles, cudaStream_t stream) {
  const int wpg = kGroup * bits / 32;
  const int64_t total = static_cast<int64_t>(tiles_bytes(K, N, bits) / 4);
  tiles_kernel<<<grid_for(total, 256), 256, 0, stream>>>(qweight, N, K / kGroup, wpg, total, tiles);
  return cudaGetLastError();
}

cudaError_t launch_wait_timeout(int64_t limit_ns, int* err, cudaStream_t stream) {
  wait_timeout_kernel<<<1, 32, 0, stream>>>(limit_ns, err);
  return cudaGetLastError();
}

}  // namespace qlin
