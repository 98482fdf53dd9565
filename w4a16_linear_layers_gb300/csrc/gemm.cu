// gemm.cu -- the W8A8 GS128 and W4A16 g128 linear layers on tcgen05.
//
// Passages: "Qwen3.8-27B-GPTQ-INT8-W8A8-GS128-PTQR" card, "Quantization
// details" (int8 x int8 compute at every decode and prefill GEMM shape, one
// weight scale per 128-wide K block); "Qwen3.8-27B-DFlash2-W4A16-g128-sym-
// GPTQ" card, property table and the apply_dense_kv_fix format table (W4A16
// GPTQ: unpack_from_int32 + group scales).
//
// GB300 (sm_103a) has no integer tcgen05 MMA, so the int8 operands are turned
// into fp16 exactly (|q| <= 128 is representable) and multiplied by
// tcgen05.mma kind::f16 with fp32 accumulation in tensor memory.  Within one
// 128-wide group every product and partial sum is an integer of magnitude at
// most 128*127*127 < 2^24, so the fp32 accumulator holds the exact integer
// group partial.
//
// Structure (one persistent block of 512 threads per SM):
//   * the output is cut into tiles of 128 features x T tokens; the MMA runs
//     with the weights as operand A (128 rows = features, held in TMEM) and
//     the tokens as operand B (T columns, in shared memory), so decode-sized
//     M only pads T up to a multiple of 16;
//   * the work is the list of (tile, group) steps; block c takes the
//     contiguous range [c*W/C, (c+1)*W/C) of the W steps (stream-K), so every
//     SM gets the same amount of weight stream whatever the shape;
//   * a tile split between blocks is finished by the last block to arrive on
//     its counter, which sums the per-block fp32 partials in ascending block
//     order (deterministic, no spin waits);
//   * warp 0 issues TMA loads into a ring of stages, warp 1 allocates TMEM and
//     issues the MMAs, the converter warps unpack weights (and, for W8A8, the
//     int8 activations) into MMA operands, the epilogue warps drain TMEM.
//
// W8A8 per group g:  D = A_g * B_g (exact integers), then acc = fma(D, s_w, acc)
// in the epilogue, ascending g; at the end y = bf16(acc * s_a).
// W4A16: A = bf16(q * s) per weight; D accumulates over all K in TMEM; y = bf16(D).
//
// Every wait is bounded (qlin_device.cuh); a wait that runs out records an
// error, aborts the block's pipeline and the block still drains its TMA
// loads and MMAs and frees its TMEM before it exits.
#include <cuda_fp16.h>
#include <cuda_bf16.h>

#include <cudaTypedefs.h>

#include <mutex>

#include "qlin_device.cuh"
#include "qlin_internal.h"

namespace qlin {
namespace {

constexpr int kThreads = 512;
constexpr int kTileF = 128;            // features per tile = MMA M
constexpr uint32_t kSmemLimit = 232448; // 227 KB opt-in shared memory per block
constexpr uint32_t kCtrlBytes = 1024;
constexpr int kMaxStages = 8;

constexpr int kModeW8A8 = 0;
constexpr int kModeP = 1;     // W8A8 pipeline, exports the group partials
constexpr int kModeW4 = 2;

template <int kMode, int T>
struct Cfg {
  static constexpr bool kW4 = kMode == kModeW4;
  static constexpr int kConvWarp0 = 4;
  static constexpr int kConvWarps = kW4 ? 8 : 4;
  static constexpr int kEpiWarp0 = kConvWarp0 + kConvWarps;
  static constexpr int kEpiWarps = 16 - kEpiWarp0;
  static constexpr int kConvThreads = 32 * kConvWarps;
  static constexpr int kEpiThreads = 32 * kEpiWarps;
  static constexpr int kWordRows = kW4 ? 16 : 32;           // int32 rows per group
  static constexpr uint32_t kWBytes = kWordRows * kTileF * 4;
  static constexpr uint32_t kABytes = kW4 ? 2u * T * 128u : T * 128u;
  static constexpr uint32_t kStageBytes = (kWBytes + kABytes + 1023u) & ~1023u;
  static constexpr uint32_t kBBytes = kW4 ? 0u : T * 256u;  // converted fp16 B, per buffer
  static constexpr uint32_t kBTotal = 2u * kBBytes;
  static constexpr uint32_t kTmemCols = (128 + 2 * T) <= 256 ? 256u : 512u;
  static constexpr uint32_t kColA = 0;      // two A buffers of 64 columns
  static constexpr uint32_t kColD = 128;    // two D buffers of T columns
  static constexpr int kEpiCols = kW4 ? T : T / 2;           // columns per epilogue thread
  static constexpr uint32_t kEmptyCount = kW4 ? kConvThreads + 1 : kConvThreads;
  static_assert(T % 16 == 0 && T >= 16 && T <= 128, "token tile");
  static_assert(kEpiCols % 8 == 0, "epilogue columns");
};

struct KParams {
  const float* s_a;
  const uint16_t* scales;
  void* out;
  int64_t M, N, G, F, W;
  float* part;
  int* counters;
  int* err;
  uint64_t limit_ns;
  int stages;
};

// Shared control block (after the stage ring and the B buffers).
struct Ctrl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t a_full[2];
  uint64_t a_empty[2];
  uint64_t d_full[2];
  uint64_t d_empty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort_flag;
  int last_flag;
};

__device__ __forceinline__ int64_t cta_of_step(int64_t s, int64_t C, int64_t W) {
  return ((s + 1) * C + W - 1) / W - 1;
}

// Four bf16 pairs of one int4 word: nibble i holds q_i + 8 for k = 8kk + i.
// Output word j holds (k = 2j, 2j+1) as bf16(q * s), rounded once.
__device__ __forceinline__ void int4x8_to_bf16x8(uint32_t w, uint32_t s2, uint32_t* out) {
  const uint32_t ev = w & 0x0F0F0F0Fu;          // nibbles 0,2,4,6 in bytes 0..3
  const uint32_t od = (w >> 4) & 0x0F0F0F0Fu;   // nibbles 1,3,5,7
  const uint32_t bias = 0x43084308u;            // bf16x2 (136, 136)
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    // bytes: ev.i, 0 (sign of ev.i), od.i, 0  ->  bf16 bits 0x43uu = 128 + u
    const uint32_t sel = static_cast<uint32_t>(i | ((8 | i) << 4) | ((4 + i) << 8) | ((12 + i) << 12));
    uint32_t v = prmt(ev, od, sel) | 0x43004300u;
    uint32_t qv;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(qv) : "r"(v), "r"(bias));      // exact: q
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(out[i]) : "r"(qv), "r"(s2));   // bf16(q * s)
  }
}

template <int kMode, int T>
__global__ void __launch_bounds__(kThreads, 1)
    qlin_gemm_kernel(const __grid_constant__ CUtensorMap tm_w,
                     const __grid_constant__ CUtensorMap tm_a, const KParams p) {
  using C = Cfg<kMode, T>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const int stages = p.stages;
  const uint32_t b_off = static_cast<uint32_t>(stages) * C::kStageBytes;
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(smem + b_off + C::kBTotal);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t nC = gridDim.x;
  const int64_t cta = blockIdx.x;
  const int64_t s0 = cta * p.W / nC;
  const int64_t s1 = (cta + 1) * p.W / nC;
  const int n_steps = static_cast<int>(s1 - s0);
  const int64_t G = p.G;
  const int64_t F = p.F;

  if (threadIdx.x == 0) {
    for (int i = 0; i < stages; ++i) {
      mbar_init(smem_u32(&ctrl->full[i]), 1);
      mbar_init(smem_u32(&ctrl->empty[i]), C::kEmptyCount);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&ctrl->a_full[i]), C::kConvThreads);
      mbar_init(smem_u32(&ctrl->a_empty[i]), 1);
      mbar_init(smem_u32(&ctrl->d_full[i]), 1);
      mbar_init(smem_u32(&ctrl->d_empty[i]), C::kEpiThreads);
    }
    mbar_init(smem_u32(&ctrl->mma_done), 1);
    ctrl->abort_flag = 0;
    ctrl->last_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&ctrl->tmem_base), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctrl->tmem_base;
  const WaitCtx ctx{p.err, &ctrl->abort_flag, p.limit_ns};
  int never_abort = 0;
  const WaitCtx drain_ctx{p.err, &never_abort, p.limit_ns};

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tm_w);
      prefetch_tmap(&tm_a);
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_a = policy_evict_last();
      int issued = 0;
      for (int j = 0; j < n_steps; ++j) {
        const int st = j % stages;
        const uint32_t ph = static_cast<uint32_t>(j / stages) & 1u;
        if (!mbar_wait(smem_u32(&ctrl->empty[st]), ph ^ 1u, ctx, 1)) break;
        const int64_t s = s0 + j;
        const int64_t tile = s / G;
        const int64_t g = s - tile * G;
        const int64_t t = tile / F;
        const int64_t f = tile - t * F;
        const uint32_t full = smem_u32(&ctrl->full[st]);
        const uint32_t dst = sbase + static_cast<uint32_t>(st) * C::kStageBytes;
        mbar_arrive_expect_tx(full, C::kWBytes + C::kABytes);
        tma_load_2d(dst, &tm_w, full, static_cast<int32_t>(f * kTileF),
                    static_cast<int32_t>(g * C::kWordRows), pol_w);
        if constexpr (C::kW4) {
          tma_load_2d(dst + C::kWBytes, &tm_a, full, static_cast<int32_t>(g * kGroup),
                      static_cast<int32_t>(t * T), pol_a);
          tma_load_2d(dst + C::kWBytes + T * 128u, &tm_a, full,
                      static_cast<int32_t>(g * kGroup + 64), static_cast<int32_t>(t * T), pol_a);
        } else {
          tma_load_2d(dst + C::kWBytes, &tm_a, full, static_cast<int32_t>(g * kGroup),
                      static_cast<int32_t>(t * T), pol_a);
        }
        ++issued;
      }
      // Every load issued must land before the block exits.
      for (int j = issued > stages ? issued - stages : 0; j < issued; ++j)
        (void)mbar_wait(smem_u32(&ctrl->full[j % stages]),
                        static_cast<uint32_t>(j / stages) & 1u, drain_ctx, 2);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16(kTileF, T, C::kW4);
      int seg = 0;
      for (int j = 0; j < n_steps; ++j) {
        const int ab = j & 1;
        const uint32_t abph = static_cast<uint32_t>(j >> 1) & 1u;
        if constexpr (C::kW4) {
          const int64_t s = s0 + j;
          const int64_t g = s % G;
          const bool first = (j == 0) || (g == 0);
          const bool last = (s == s1 - 1) || (g == G - 1);
          const int st = j % stages;
          const uint32_t ph = static_cast<uint32_t>(j / stages) & 1u;
          const int db = seg & 1;
          const uint32_t dbph = static_cast<uint32_t>(seg >> 1) & 1u;
          if (!mbar_wait(smem_u32(&ctrl->full[st]), ph, ctx, 3)) break;
          if (!mbar_wait(smem_u32(&ctrl->a_full[ab]), abph, ctx, 4)) break;
          if (first && !mbar_wait(smem_u32(&ctrl->d_empty[db]), dbph ^ 1u, ctx, 5)) break;
          tc_fence_after();
          const uint32_t xb = sbase + static_cast<uint32_t>(st) * C::kStageBytes + C::kWBytes;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint64_t bdesc =
                smem_desc(xb + static_cast<uint32_t>(ks >> 2) * (T * 128u) +
                              static_cast<uint32_t>(ks & 3) * 32u,
                          16u, 1024u, 2u);
            mma_ts(tmem + C::kColD + db * T, tmem + C::kColA + ab * 64 + ks * 8, bdesc, idesc,
                   (first && ks == 0) ? 0u : 1u);
          }
          tc_commit(smem_u32(&ctrl->a_empty[ab]));
          tc_commit(smem_u32(&ctrl->empty[st]));
          if (last) {
            tc_commit(smem_u32(&ctrl->d_full[db]));
            ++seg;
          }
        } else {
          if (!mbar_wait(smem_u32(&ctrl->a_full[ab]), abph, ctx, 3)) break;
          if (!mbar_wait(smem_u32(&ctrl->d_empty[ab]), abph ^ 1u, ctx, 4)) break;
          tc_fence_after();
          const uint32_t bb = sbase + b_off + static_cast<uint32_t>(ab) * C::kBBytes;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            // canonical K-major, no swizzle: core matrices of 8 rows x 16 B;
            // LBO = 128 B between K-adjacent core matrices, SBO = 2048 B
            // between 8-row groups.
            const uint64_t bdesc = smem_desc(bb + static_cast<uint32_t>(ks) * 256u, 128u, 2048u, 0u);
            mma_ts(tmem + C::kColD + ab * T, tmem + C::kColA + ab * 64 + ks * 8, bdesc, idesc,
                   ks > 0 ? 1u : 0u);
          }
          tc_commit(smem_u32(&ctrl->a_empty[ab]));
          tc_commit(smem_u32(&ctrl->d_full[ab]));
        }
      }
      tc_commit(smem_u32(&ctrl->mma_done));
      (void)mbar_wait(smem_u32(&ctrl->mma_done), 0u, drain_ctx, 6);
    }
  } else if (warp >= C::kConvWarp0 && warp < C::kEpiWarp0) {
    // ------------------------------------------------------------ converters
    const int ct = threadIdx.x - 32 * C::kConvWarp0;
    const int r = ct & 127;                      // row of A = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    for (int j = 0; j < n_steps; ++j) {
      const int st = j % stages;
      const uint32_t ph = static_cast<uint32_t>(j / stages) & 1u;
      const int ab = j & 1;
      const uint32_t abph = static_cast<uint32_t>(j >> 1) & 1u;
      bool ok = mbar_wait(smem_u32(&ctrl->full[st]), ph, ctx, 7);
      if (ok) ok = mbar_wait(smem_u32(&ctrl->a_empty[ab]), abph ^ 1u, ctx, 8);
      if (!named_bar_and(3, C::kConvThreads, ok)) break;
      tc_fence_after();
      const uint8_t* stage = smem + static_cast<uint32_t>(st) * C::kStageBytes;
      const uint32_t* wsm = reinterpret_cast<const uint32_t*>(stage);
      const uint32_t acol = tmem + lane_off + C::kColA + ab * 64;
      if constexpr (C::kW4) {
        const int kh = ct >> 7;                  // which half of the group's K
        const int64_t s = s0 + j;
        const int64_t tile = s / G;
        const int64_t g = s - tile * G;
        const int64_t n = (tile % F) * kTileF + r;
        uint32_t s2 = 0;
        if (n < p.N) {
          const uint32_t sb = p.scales[g * p.N + n];
          s2 = sb | (sb << 16);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t v[16];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            int4x8_to_bf16x8(wsm[(kh * 8 + h * 4 + i) * kTileF + r], s2, v + 4 * i);
          tmem_st16(acol + kh * 32 + h * 16, v);
        }
      } else {
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          uint32_t v[16];
#pragma unroll
          for (int i = 0; i < 8; ++i)
            biased_u8x4_to_f16x4(wsm[(h * 8 + i) * kTileF + r], v[2 * i], v[2 * i + 1]);
          tmem_st16(acol + h * 16, v);
        }
        // int8 activations (128-byte swizzled TMA tile, T rows x 128 B) ->
        // fp16 canonical layout in B buffer ab.
        const uint8_t* araw = stage + C::kWBytes;
        uint8_t* bbuf = smem + b_off + static_cast<uint32_t>(ab) * C::kBBytes;
#pragma unroll
        for (int i = 0; i < T / 16; ++i) {
          const int x = ct + 128 * i;
          const int cc = x / T;
          const int rr = x - cc * T;
          const uint4 raw =
              *reinterpret_cast<const uint4*>(araw + rr * 128 + ((cc ^ (rr & 7)) << 4));
          uint4 o0, o1;
          biased_u8x4_to_f16x4(raw.x ^ 0x80808080u, o0.x, o0.y);
          biased_u8x4_to_f16x4(raw.y ^ 0x80808080u, o0.z, o0.w);
          biased_u8x4_to_f16x4(raw.z ^ 0x80808080u, o1.x, o1.y);
          biased_u8x4_to_f16x4(raw.w ^ 0x80808080u, o1.z, o1.w);
          uint8_t* dst = bbuf + (rr >> 3) * 2048 + (rr & 7) * 16 + cc * 256;
          *reinterpret_cast<uint4*>(dst) = o0;
          *reinterpret_cast<uint4*>(dst + 128) = o1;
        }
        fence_proxy_async_smem();
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(smem_u32(&ctrl->empty[st]));
      mbar_arrive(smem_u32(&ctrl->a_full[ab]));
    }
  } else if (warp >= C::kEpiWarp0) {
    // ------------------------------------------------------------ epilogue
    const int et = threadIdx.x - 32 * C::kEpiWarp0;
    const int r = (warp & 3) * 32 + lane;        // TMEM lane = feature in tile
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int colbase = C::kW4 ? 0 : ((warp - C::kEpiWarp0) >> 2) * (T / 2);
    const int64_t M = p.M, N = p.N;
    const int64_t first_tile = s0 / G;
    uint16_t* y = static_cast<uint16_t*>(p.out);

    if constexpr (!C::kW4) {
      float acc[C::kEpiCols];
      int64_t seg_g0 = 0;
      for (int j = 0; j < n_steps; ++j) {
        const int64_t s = s0 + j;
        const int64_t tile = s / G;
        const int64_t g = s - tile * G;
        const int64_t t = tile / F;
        const int64_t f = tile - t * F;
        const int64_t n = f * kTileF + r;
        if (j == 0 || g == 0) {
          seg_g0 = g;
#pragma unroll
          for (int c = 0; c < C::kEpiCols; ++c) acc[c] = 0.0f;
        }
        const int b = j & 1;
        const uint32_t bph = static_cast<uint32_t>(j >> 1) & 1u;
        float sw = 0.0f;
        if (kMode == kModeW8A8 && n < N)
          sw = __half2float(__ushort_as_half(p.scales[g * N + n]));
        const bool ok = mbar_wait(smem_u32(&ctrl->d_full[b]), bph, ctx, 9);
        if (!named_bar_and(2, C::kEpiThreads, ok)) break;
        tc_fence_after();
        const uint32_t dcol = tmem + lane_off + C::kColD + b * T + colbase;
        constexpr int kCh = C::kEpiCols < 16 ? C::kEpiCols : 16;
#pragma unroll
        for (int c0 = 0; c0 < C::kEpiCols; c0 += kCh) {
          uint32_t v[kCh];
          if constexpr (kCh == 16) tmem_ld16(dcol + c0, v);
          else tmem_ld8(dcol + c0, v);
          tmem_wait_ld();
          if constexpr (kMode == kModeP) {
            int32_t* P = static_cast<int32_t*>(p.out);
#pragma unroll
            for (int c = 0; c < kCh; ++c) {
              const int64_t m = t * T + colbase + c0 + c;
              if (m < M && n < N)
                P[(g * M + m) * N + n] = static_cast<int32_t>(__uint_as_float(v[c]));
            }
          } else {
#pragma unroll
            for (int c = 0; c < kCh; ++c) acc[c0 + c] = fmaf(__uint_as_float(v[c]), sw, acc[c0 + c]);
          }
        }
        tc_fence_before();
        mbar_arrive(smem_u32(&ctrl->d_empty[b]));

        if constexpr (kMode == kModeP) {
          continue;
        } else {
          if (!(s == s1 - 1 || g == G - 1)) continue;

          // ---- end of this block's segment of the tile
          const bool full_tile = (seg_g0 == 0) && (g == G - 1);
          bool write = full_tile;
          if (!full_tile) {
            const int slot = (tile == first_tile) ? 0 : 1;
            float* mine = p.part + ((cta * 2 + slot) * T) * kTileF;
#pragma unroll
            for (int c = 0; c < C::kEpiCols; ++c) mine[(colbase + c) * kTileF + r] = acc[c];
            __threadfence();
            named_bar_sync(1, C::kEpiThreads);
            const int64_t c_first = cta_of_step(tile * G, nC, p.W);
            const int64_t c_last = cta_of_step(tile * G + G - 1, nC, p.W);
            if (et == 0) {
              const int old = atomicAdd(&p.counters[tile], 1);
              ctrl->last_flag = (old == static_cast<int>(c_last - c_first)) ? 1 : 0;
            }
            named_bar_sync(1, C::kEpiThreads);
            write = ctrl->last_flag != 0;
            if (write) {
              __threadfence();
#pragma unroll
              for (int c = 0; c < C::kEpiCols; ++c) acc[c] = 0.0f;
              for (int64_t cc = c_first; cc <= c_last; ++cc) {
                const int slot2 = ((cc * p.W / nC) / G == tile) ? 0 : 1;
                const float* pp = p.part + ((cc * 2 + slot2) * T) * kTileF;
#pragma unroll
                for (int c = 0; c < C::kEpiCols; ++c) acc[c] += __ldcg(pp + (colbase + c) * kTileF + r);
              }
              if (et == 0) p.counters[tile] = 0;
            }
          }
          if (write && n < N) {
#pragma unroll
            for (int c = 0; c < C::kEpiCols; ++c) {
              const int64_t m = t * T + colbase + c;
              if (m < M)
                y[m * N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[c] * __ldg(p.s_a + m)));
            }
          }
        }
      }
    } else {
      int seg = 0;
      int64_t seg_g0 = 0;
      for (int j = 0; j < n_steps; ++j) {
        const int64_t s = s0 + j;
        const int64_t tile = s / G;
        const int64_t g = s - tile * G;
        if (j == 0 || g == 0) seg_g0 = g;
        if (!(s == s1 - 1 || g == G - 1)) continue;
        const int64_t t = tile / F;
        const int64_t f = tile - t * F;
        const int64_t n = f * kTileF + r;
        const int db = seg & 1;
        const uint32_t dbph = static_cast<uint32_t>(seg >> 1) & 1u;
        ++seg;
        const bool ok = mbar_wait(smem_u32(&ctrl->d_full[db]), dbph, ctx, 10);
        if (!named_bar_and(2, C::kEpiThreads, ok)) break;
        tc_fence_after();
        const uint32_t dcol = tmem + lane_off + C::kColD + db * T;
        const bool full_tile = (seg_g0 == 0) && (g == G - 1);
        if (full_tile) {
#pragma unroll
          for (int ch = 0; ch < T / 16; ++ch) {
            uint32_t v[16];
            tmem_ld16(dcol + ch * 16, v);
            tmem_wait_ld();
            if (n < N) {
#pragma unroll
              for (int c = 0; c < 16; ++c) {
                const int64_t m = t * T + ch * 16 + c;
                if (m < M) y[m * N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(v[c])));
              }
            }
          }
          tc_fence_before();
          mbar_arrive(smem_u32(&ctrl->d_empty[db]));
        } else {
          const int slot = (tile == first_tile) ? 0 : 1;
          float* mine = p.part + ((cta * 2 + slot) * T) * kTileF;
#pragma unroll
          for (int ch = 0; ch < T / 16; ++ch) {
            uint32_t v[16];
            tmem_ld16(dcol + ch * 16, v);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 16; ++c) mine[(ch * 16 + c) * kTileF + r] = __uint_as_float(v[c]);
          }
          tc_fence_before();
          mbar_arrive(smem_u32(&ctrl->d_empty[db]));
          __threadfence();
          named_bar_sync(1, C::kEpiThreads);
          const int64_t c_first = cta_of_step(tile * G, nC, p.W);
          const int64_t c_last = cta_of_step(tile * G + G - 1, nC, p.W);
          if (et == 0) {
            const int old = atomicAdd(&p.counters[tile], 1);
            ctrl->last_flag = (old == static_cast<int>(c_last - c_first)) ? 1 : 0;
          }
          named_bar_sync(1, C::kEpiThreads);
          if (ctrl->last_flag) {
            __threadfence();
#pragma unroll
            for (int ch = 0; ch < T / 16; ++ch) {
              float sum[16];
#pragma unroll
              for (int c = 0; c < 16; ++c) sum[c] = 0.0f;
              for (int64_t cc = c_first; cc <= c_last; ++cc) {
                const int slot2 = ((cc * p.W / nC) / G == tile) ? 0 : 1;
                const float* pp = p.part + ((cc * 2 + slot2) * T) * kTileF;
#pragma unroll
                for (int c = 0; c < 16; ++c) sum[c] += __ldcg(pp + (ch * 16 + c) * kTileF + r);
              }
              if (n < N) {
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                  const int64_t m = t * T + ch * 16 + c;
                  if (m < M) y[m * N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(sum[c]));
                }
              }
            }
            if (et == 0) p.counters[tile] = 0;
          }
        }
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ------------------------------------------------------------------- host

using EncodeFn = PFN_cuTensorMapEncodeTiled_v12000;

EncodeFn encode_fn() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(ptr);
  });
  return fn;
}

bool make_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner,
                 uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                 CUtensorMapSwizzle swz) {
  EncodeFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int kMode, int T>
cudaError_t launch_t(const GemmArgs& a, const GemmPlan& pl, int* err, cudaStream_t stream) {
  using C = Cfg<kMode, T>;
  CUtensorMap tw, ta;
  const uint64_t words_rows = static_cast<uint64_t>(a.K) / (C::kW4 ? 8 : 4);
  if (!make_map_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_INT32, a.qweight, a.N, words_rows,
                   static_cast<uint64_t>(a.N) * 4, kTileF, C::kWordRows,
                   CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  bool ok;
  if constexpr (C::kW4)
    ok = make_map_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.act, a.K, a.M,
                     static_cast<uint64_t>(a.K) * 2, 64, T, CU_TENSOR_MAP_SWIZZLE_128B);
  else
    ok = make_map_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.act, a.K, a.M,
                     static_cast<uint64_t>(a.K), 128, T, CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) return cudaErrorInvalidValue;

  const uint32_t fixed = 1024 + C::kBTotal + kCtrlBytes;
  int stages = static_cast<int>((kSmemLimit - fixed) / C::kStageBytes);
  if (stages > kMaxStages) stages = kMaxStages;
  const uint32_t smem = fixed + static_cast<uint32_t>(stages) * C::kStageBytes;

  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(qlin_gemm_kernel<kMode, T>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(kSmemLimit));
  });
  if (attr_err != cudaSuccess) return attr_err;

  KParams kp;
  kp.s_a = a.s_a;
  kp.scales = a.scales;
  kp.out = a.out;
  kp.M = a.M;
  kp.N = a.N;
  kp.G = pl.G;
  kp.F = pl.F;
  kp.W = pl.steps;
  kp.counters = static_cast<int*>(a.workspace);
  kp.part = reinterpret_cast<float*>(static_cast<uint8_t*>(a.workspace) + pl.counter_bytes);
  kp.err = err;
  kp.limit_ns = kWaitLimitNs;
  kp.stages = stages;
  qlin_gemm_kernel<kMode, T><<<static_cast<unsigned>(pl.ctas), kThreads, smem, stream>>>(tw, ta, kp);
  return cudaGetLastError();
}

template <int kMode>
cudaError_t launch_mode(const GemmArgs& a, const GemmPlan& pl, int* err, cudaStream_t stream) {
  switch (pl.T) {
    case 16: return launch_t<kMode, 16>(a, pl, err, stream);
    case 32: return launch_t<kMode, 32>(a, pl, err, stream);
    case 64: return launch_t<kMode, 64>(a, pl, err, stream);
    case 96: return launch_t<kMode, 96>(a, pl, err, stream);
    default: return launch_t<kMode, 128>(a, pl, err, stream);
  }
}

}  // namespace

GemmPlan plan_gemm(int64_t M, int64_t N, int64_t K, int sm_count) {
  GemmPlan p{};
  p.T = M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : M <= 96 ? 96 : 128;
  p.F = (N + kTileF - 1) / kTileF;
  p.TT = (M + p.T - 1) / p.T;
  p.G = K / kGroup;
  p.steps = p.TT * p.F * p.G;
  p.ctas = p.steps < sm_count ? p.steps : sm_count;
  if (p.ctas < 1) p.ctas = 1;
  p.counter_bytes = ((static_cast<size_t>(p.TT * p.F) * sizeof(int)) + 255) & ~static_cast<size_t>(255);
  p.workspace_bytes = p.counter_bytes + static_cast<size_t>(p.ctas) * 2 * p.T * kTileF * sizeof(float);
  return p;
}

cudaError_t launch_gemm(const GemmArgs& a, const GemmPlan& p, int* err, cudaStream_t stream) {
  switch (a.mode) {
    case GemmMode::kW8A8: return launch_mode<kModeW8A8>(a, p, err, stream);
    case GemmMode::kW8A8Partials: return launch_mode<kModeP>(a, p, err, stream);
    default: return launch_mode<kModeW4>(a, p, err, stream);
  }
}

}  // namespace qlin
