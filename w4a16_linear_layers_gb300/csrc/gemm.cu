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
// Structure (one persistent block of 512, 640 or 768 threads per SM):
//   * the output is cut into tiles of 128 features x T tokens; the MMA runs
//     with the weights as operand A (128 rows = features, converted by
//     threads straight into TMEM) and the tokens as operand B (T columns,
//     16-bit, 128-byte swizzled in shared memory), so decode-sized M only
//     pads T up to a multiple of 16;
//   * W4A16 tokens (bf16) land by TMA directly in the operand layout; W8A8
//     tokens of tiles up to 32 land as int8 tiles and the converter group of
//     the step expands them exactly to fp16 beside the weights it converts
//     (half the bytes from L2, and no extra kernel between act-quant and the
//     GEMM); larger W8A8 tiles read 16-bit codes by TMA: the caller's fp16
//     codes, or an exact fp16 image of int8 codes written by a small pre-pass
//     kernel;
//   * the work is the list of (tile, group) steps; block c takes the
//     contiguous range [c*W/C, (c+1)*W/C) of the W steps (stream-K), so every
//     SM gets the same amount of weight stream whatever the shape;
//   * a tile split between blocks is finished by the last block to arrive on
//     its counter, which sums the per-block fp32 partials in ascending block
//     order (deterministic); at W8A8 tiles of 64 and more the tile's first
//     contributor arrives only after its last step and, when it is not the
//     last, publishes afterwards, so the finisher waits (bounded) for its
//     flag -- on a block that has already arrived;
//   * roles: warp 0 streams weights by TMA, warp 2 streams activations and
//     group scales, warps 1 and 3 issue the MMAs of alternate steps (one
//     thread's issue rate is below what the weight stream needs), warps 4-11
//     convert weights into TMEM (and W8A8 tokens into fp16), warps 12 and
//     up drain TMEM (one per TMEM lane quarter for W8A8 tiles of 32 and
//     fewer, two otherwise, three at 96-token tiles).
//
// W8A8 per group g:  D = A_g * B_g (exact integers), then acc = fma(D, s_w, acc)
// in the epilogue, ascending g; at the end y = bf16(acc * s_a).
// W4A16: A = bf16(q * s) per weight; D accumulates over all K in TMEM (one
// accumulator per MMA issuer, summed in the epilogue); y = bf16(D).
//
// Every wait is bounded (qlin_device.cuh); a wait that runs out records an
// error, aborts the block's pipeline and the block still drains its TMA
// loads and MMAs and frees its TMEM before it exits.
//
// Launches use programmatic dependent launch: a kernel lets the next one start
// early and every kernel waits for its predecessor (griddepcontrol.wait)
// before it touches anything the predecessor may produce or consume
// (activations, outputs, workspace).  Weights and scales are read without
// waiting; the packer, which writes weights, never lets its successor start
// early.
#include <cuda_fp16.h>
#include <cuda_bf16.h>

#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "qlin_device.cuh"
#include "qlin_internal.h"

namespace qlin {
namespace {

constexpr int kTileF = 128;            // features per tile = MMA M
constexpr uint32_t kSmemLimit = 232448; // 227 KB opt-in shared memory per block
constexpr uint32_t kCtrlBytes = 1024;
constexpr int kMaxStages = 16;           // weight ring slots
constexpr int kMaxXSlots = 16;           // activation ring slots
constexpr size_t kCounterBytes = 5120;   // int counters for up to 1024 blocks, then
                                         // the argmax keys (kArgmaxKeysOffset)
constexpr uint32_t kArgBytes = 4096;     // shared argmax keys: [4 lane quarters][128 tokens]
constexpr int64_t kMinSteps = 8;          // minimum (tile, group) steps per block
constexpr int kScaleChunk = 8;            // groups of scales per TMA load
constexpr int kPreW = 3;                  // weight loads issued before the first activations
constexpr int64_t kBandMinTiles = 6;      // token tiles from which whole tiles go in bands
constexpr int64_t kBandBytes = 48ll << 20;   // activation bytes of one band

constexpr int kModeW8A8 = 0;
constexpr int kModeP = 1;     // W8A8 pipeline, exports the group partials
constexpr int kModeW4 = 2;
constexpr int kModeW8A16 = 3;   // int8 weight-only: group-32, group-128 or per-column scales

template <int kMode, int T, int GPS = 1>
struct Cfg {
  // weight-only formats (W4A16, W8A16): bf16 tokens, scales applied by the
  // converters, the whole K accumulated in TMEM
  static constexpr bool kWO = kMode == kModeW4 || kMode == kModeW8A16;
  static constexpr bool kInt4 = kMode == kModeW4;
  // 128-wide K groups per pipeline step.  W4A16 at token tiles up to 32 takes
  // two: a step then carries 16 KB of weights like the 8-bit formats, which
  // halves the fixed per-step cost (synchronisation, MMA issue) per byte.  At
  // 64-token tiles the larger activation slots halve the weight bytes in
  // flight, which costs more than it saves on short ranges: there two-group
  // steps are taken only when every block gets at least 16 of them.
  static constexpr int kGPS = GPS;
  static_assert(GPS == 1 || (GPS == 2 && kInt4 && T <= 64), "two-group steps: W4A16, T <= 64");
  // warps 0..3: control (0 weight TMA, 1 TMEM owner + MMA issuer, 2 activation
  //             and scale TMA, 3 MMA issuer)
  // warps 4..11: converters, two groups of four taking alternate steps (each
  //              converts a whole 128-wide K group; warp w serves TMEM lanes
  //              32*(w%4)..)
  // warps 12..: epilogue, kEpiPerQ warps per TMEM lane quarter, each
  //              draining T / kEpiPerQ token columns of the accumulator, all
  //              of them with one batch of TMEM loads (at most 32 columns, so
  //              the loaded values and the running sums fit in registers).
  //              W8A8 token tiles of 32 and fewer take one warp per quarter:
  //              512 threads leave 128 registers a thread instead of 96 (no
  //              spills) and four fewer warps compete for issue slots, which
  //              ran the decode shapes 4-5% faster; the weight-only formats,
  //              whose epilogue drains once per segment, measured no gain.
  static constexpr int kConvWarp0 = 4;
  static constexpr int kConvWarps = 8;
  static constexpr int kEpiWarp0 = 12;
  static constexpr int kEpiPerQ = T > 64 ? 3 : (T <= 32 && !kWO ? 1 : 2);
  static constexpr int kEpiWarps = 4 * kEpiPerQ;
  static constexpr int kConvThreads = 32 * kConvWarps;
  static constexpr int kEpiThreads = 32 * kEpiWarps;
  static constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps);
  static constexpr int kWordRows = (kInt4 ? 16 : 32) * GPS;  // int32 rows per step
  static constexpr uint32_t kWBytes = kWordRows * kTileF * 4;
  static constexpr uint32_t kABytes = 2u * T * 128u * GPS;   // 64-wide 16-bit halves
  static constexpr int kACols = 64 * GPS;                     // TMEM columns per A buffer
  // Weights and activations travel in rings of their own, so neither stream
  // waits for the other's consumer.  A weight slot is freed as soon as the
  // converters have read it into registers.
  //   W4A16: bf16 activation tiles land by TMA in the MMA's operand layout; a
  //   slot is freed when the MMAs that read it have completed.
  //   W8A8, T <= 32: int8 activation tiles land by TMA in a staging ring
  //   (freed by the converters) and the converter group of the step expands
  //   them exactly to fp16 in the operand slot that pairs with its A buffer.
  //   W8A8, T >= 64: that expansion would add 24-36 KB of shared-memory
  //   traffic and a quarter of the converters' instructions per step; the
  //   caller's fp16 codes, or an exact fp16 image written once by a pre-pass
  //   kernel, land like W4A16's tiles.
  // The first ring in each case is deep enough to cover the L2 latency seen
  // while the weight stream keeps HBM busy.
  static constexpr uint32_t kStageBytes = kWBytes;
  static constexpr uint32_t kXiBytes = static_cast<uint32_t>(T) * 128u;   // int8 tile
  static constexpr int kXiRaw = static_cast<int>(32768u / kXiBytes);
  static constexpr bool kXConv = !kWO && T <= 32;
  static constexpr int kXiSlots = !kXConv ? 0 : (kXiRaw < 4 ? 4 : (kXiRaw > kMaxXSlots ? kMaxXSlots : kXiRaw));
  static constexpr int kXSlotsRaw = static_cast<int>(65536u / kABytes);
  static constexpr int kXSlotsW4 = kXSlotsRaw < 4 ? 4 : (kXSlotsRaw > kMaxXSlots ? kMaxXSlots : kXSlotsRaw);
  static constexpr int kIssuers = 2;
  // W4A16 accumulates a whole segment in TMEM: one accumulator per issuer
  // and segment buffer (two segment buffers while they fit).
  static constexpr int kSegBufs = kWO ? (T <= 96 ? 2 : 1) : 0;
  static constexpr int kW4DCols = kWO ? kSegBufs * kIssuers * T : 0;
  // A (64 TMEM columns) and, for W8A8, D (T columns) buffers in flight
  // between the converters, the MMA issuers and the epilogue.
  // W8A8 sizes the A buffers (converter -> MMA) and the D buffers (MMA ->
  // epilogue) separately: the epilogue loop (MMA completion, TMEM drain,
  // release) is the long one, so small token tiles get many D buffers.
  // Token tiles of 64 and more keep two A buffers (one per converter group)
  // and give the columns to D buffers: six at 64 tokens, four at 96.  There
  // the D ring sets the pace (each buffer goes round MMA completion, the
  // epilogue's wake-up, drain and release, and the issuer's wake-up), while
  // a converter group loads its next step's weights before it waits for its
  // A buffer, so only the TMEM stores sit in the A loop.
  static constexpr int kNumBufRaw = kWO ? (512 - kW4DCols) / kACols : (T <= 32 ? 4 : 2);
  // An even count keeps every A buffer with one converter group and one
  // issuer (steps alternate between the two of each).
  static constexpr int kNumBufCap = kNumBufRaw < 6 ? kNumBufRaw : 6;
  static constexpr int kNumBuf = kNumBufCap - (kNumBufCap & 1);
  static constexpr int kNumDFit = kWO ? 1 : (512 - 64 * kNumBuf) / T;
  static constexpr int kNumDRaw = kNumDFit < 16 ? kNumDFit : 16;
  // W8A8 with at least as many D buffers as A buffers commits once per step,
  // on the step's D buffer: that completion also frees the step's A buffer
  // and fp16 operand slot (slot i pairs with A buffer i), which the
  // converters wait for before they refill both (ND - NA even: see the
  // waits of the converters).  With fewer D buffers than A buffers (96-token
  // tiles) the A buffers are freed by commits of their own, as in the
  // weight-only formats.
  static constexpr int kNumDEven = kNumDRaw - ((kNumDRaw - kNumBuf) & 1);
  static constexpr int kNumD = kWO ? 1 : (kNumDRaw >= kNumBuf ? kNumDEven : kNumDRaw);
  static constexpr bool kACommit = kWO || kNumD < kNumBuf;
  static constexpr int kXSlots = kXConv ? kNumBuf : kXSlotsW4;
  static_assert(kACommit || (kNumD >= kNumBuf && (kNumD - kNumBuf) % 2 == 0),
                "one commit per step needs ND >= NA with ND - NA even");
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColA = 0;
  static constexpr uint32_t kColD = kACols * kNumBuf;
  static constexpr int kEpiCols = T / kEpiPerQ;              // columns per epilogue thread
  // a weight slot is released by the four warps of one converter group
  static constexpr uint32_t kEmptyCount = kConvWarps / 2;
  // Group scales travel by TMA into a ring of their own (kScaleChunk groups x
  // 128 x 16-bit per slot), read by the epilogue (W8A8) or the converters
  // (W4A16).
  static constexpr bool kScales = kMode != kModeP;
  static constexpr int kScaleSlots = 4;
  // W8A16 group-32 scales bring 4 rows per 128-wide group
  static constexpr uint32_t kScaleRowsMax = (kMode == kModeW8A16 ? 4 : GPS) * kScaleChunk;
  static constexpr uint32_t kScaleSlotBytes = kScaleRowsMax * 256u;
  static constexpr uint32_t kScaleBytes = kScales ? kScaleSlots * kScaleSlotBytes : 0u;
  static_assert(T % 16 == 0 && T >= 16 && T <= 128, "token tile");
  static_assert(T % kEpiPerQ == 0 && kEpiCols % 8 == 0 && kEpiCols <= 32, "epilogue columns");
  static_assert(kNumBuf >= 2, "double buffering at least");
  static_assert(kColD + (kWO ? kW4DCols : kNumD * T) <= kTmemCols, "TMEM budget");
  static_assert(kWO || kNumD >= 2, "double buffering at least");
  static_assert(kConvThreads == 256 && kThreads <= 1024, "warp roles");
};

constexpr int kBufMax = 6;     // A buffers
constexpr int kDBufMax = 16;   // D buffers

struct KParams {
  unsigned long long* amax_keys;   // greedy-argmax variant, else nullptr
  // Weights in the tile layout (qlin_pack_tiles): tile (f, g) of 128 features
  // x one 128-wide K group is a contiguous block of WORDS x 128 int32
  // (WORDS = 32 for 8-bit, 16 for 4-bit), tiles ordered by f then g, each
  // brought in by one bulk copy.  nullptr: the GPTQ [K*bits/32, N] words by
  // 2D tensor-map tiles.
  const uint8_t* wtiles;
  int64_t groups;                  // K / 128 (tile columns per feature tile)
  int s_rps;                       // W8A16: scale rows per 128-wide group (4, 1; 0 = one row)
  uint32_t s_tx;                   // bytes of one scale-chunk load
  const float* s_a;
  void* out;
  int64_t M, N, G, F, W;
  int64_t TT;                      // token tiles
  int64_t band;                    // banded-tile schedule: token tiles per band; 0 = stream-K
  float* part;
  int* counters;
  int* err;
  uint64_t limit_ns;
  int stages;
};

// Shared control block (after the stage ring and the scale ring).
struct Ctrl {
  uint64_t wfull[kMaxStages];   // the slot's weights landed
  uint64_t empty[kMaxStages];   // the slot's weights are in TMEM
  uint64_t xfull[kMaxXSlots];   // W4A16: the slot's activations landed;
                                // W8A8: the staging slot's int8 tile landed
  uint64_t xempty[kMaxXSlots];  // W4A16: the MMAs reading the slot completed;
                                // W8A8: the converters read the staging slot
  uint64_t a_full[kBufMax];
  uint64_t a_empty[kBufMax];
  uint64_t d_full[kDBufMax];
  uint64_t d_empty[kDBufMax];
  uint64_t s_full[4];
  uint64_t s_empty[4];
  uint64_t mma_done;
  uint64_t x_go;                // the first activation loads are queued
  uint64_t fix_full;            // split-tile partials landed in shared memory
  uint32_t tmem_base;
  int abort_flag;
  int last_flag;
};

static_assert(sizeof(Ctrl) <= kCtrlBytes, "control block");

__device__ __forceinline__ int64_t cta_of_step(int64_t s, int64_t C, int64_t W) {
  return ((s + 1) * C + W - 1) / W - 1;
}

// Walks a block's (tile, group) steps: g is the group, f the feature tile
// and t the token tile of the current step.  Two schedules:
//  * stream-K (band == 0): the block's contiguous range of the step list,
//    tiles in token-tile-major order, a range may start and end mid-tile;
//  * banded tiles (band > 0, batches of many token tiles): block c takes whole
//    tiles c, c + C, c + 2C, ... of an order that walks bands of `band` token
//    tiles: within a band, feature tile by feature tile, every token tile of
//    the band.  The blocks running at one time then share a few feature
//    tiles' weights and one band's activations, which L2 holds, instead of
//    each block streaming every weight tile once per token tile from DRAM.
struct StepIter {
  int64_t G, F, TT, band, C;
  int64_t g, f, t, q;   // q: the tile's index in the schedule's order
  __device__ __forceinline__ StepIter(const KParams& p, int64_t s0)
      : G(p.G), F(p.F), TT(p.TT), band(p.band), C(gridDim.x) {
    if (band > 0) {
      g = 0;
      q = blockIdx.x;
      place();
    } else {
      q = s0 / G;
      g = s0 - q * G;
      t = q / F;
      f = q - t * F;
    }
  }
  __device__ __forceinline__ void place() {   // banded order: q -> (f, t)
    const int64_t b = q / (band * F);
    const int64_t r = q - b * band * F;
    const int64_t rows = (TT - b * band) < band ? (TT - b * band) : band;
    f = r / rows;
    t = b * band + (r - f * rows);
  }
  __device__ __forceinline__ int64_t tile() const { return band > 0 ? q : t * F + f; }
  __device__ __forceinline__ void next() {
    if (++g == G) {
      g = 0;
      if (band > 0) {
        q += C;
        if (q < TT * F) place();
      } else if (++f == F) {
        f = 0;
        ++t;
      }
    }
  }
};

// Position in a ring of n slots: slot index and the parity of its phase.
struct Ring {
  int n, slot = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ explicit Ring(int n_) : n(n_) {}
  __device__ __forceinline__ void next() {
    if (++slot == n) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

// Scale chunks: a segment (one block's run of groups of one tile) is cut into
// chunks of kScaleChunk groups, each brought in by one TMA load.
struct ChunkIter {
  int cg = 0;      // group offset inside the current segment
  int ci = -1;     // chunk counter
  __device__ __forceinline__ bool begin(bool seg_first) {
    if (seg_first) cg = 0;
    const bool starts = (cg % kScaleChunk) == 0;
    if (starts) ++ci;
    return starts;
  }
  __device__ __forceinline__ int row() const { return cg % kScaleChunk; }
  __device__ __forceinline__ bool ends(bool seg_last) const {
    return seg_last || (cg % kScaleChunk) == kScaleChunk - 1;
  }
  __device__ __forceinline__ void advance() { ++cg; }
};

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

// N consecutive TMEM columns (N a multiple of 8) of this warp's 32 lanes into
// v, issued as one batch; the caller waits with tmem_wait_ld.
template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t* v) {
  static_assert(N % 8 == 0, "columns");
#pragma unroll
  for (int c = 0; c + 16 <= N; c += 16) tmem_ld16(taddr + c, v + c);
  if constexpr (N % 16 == 8) tmem_ld8(taddr + (N - 8), v + (N - 8));
}

// One step's weights into a ring slot: kWordRows x 128 int32, either one
// contiguous bulk copy from the tile layout (the step's GPS groups are
// consecutive tiles) or a 2D tensor-map tile of the GPTQ words.
template <class C>
__device__ __forceinline__ void load_weights(uint32_t dst, const CUtensorMap* tm_w, const KParams& p,
                                             const StepIter& it, uint32_t full, uint64_t pol) {
  if (p.wtiles != nullptr) {
    const int64_t tile = it.f * p.groups + it.g * C::kGPS;
    bulk_load_hint(dst, p.wtiles + tile * static_cast<int64_t>(C::kWBytes / C::kGPS), C::kWBytes, full,
                   pol);
  } else {
    tma_load_2d(dst, tm_w, full, static_cast<int32_t>(it.f * kTileF),
                static_cast<int32_t>(it.g * C::kWordRows), pol);
  }
}

// All lanes of the warp agree on a wait's outcome.
__device__ __forceinline__ bool warp_all(bool ok) { return __all_sync(0xFFFFFFFFu, ok); }

// A tile whose K was split across blocks is finished by the last of its
// blocks to arrive on the arrival counter of its first contributing block.
// - A block whose range starts inside the tile (or lies inside it) publishes
//   its fp32 partial right away and counts its arrival (split_publish), but
//   looks at the count only after its last step, so no block stalls
//   mid-stream on the atomic's round trip.  Ordering: the epilogue threads'
//   partial stores are ordered before thread 0's release by the barrier.
// - For W8A8 at token tiles of 64 and more (kLate), the tile's first contributor,
//   whose range ends inside the tile, counts its arrival only after its last
//   step (split_finish).  If that arrival completes the count it finishes
//   the tile from its own registers; if not, it publishes its partial and
//   then raises kSplitPublished on the counter with release semantics, and
//   the finisher waits for that flag before it reads the partial.  (At 96
//   tokens this ran the decode launches 3.5% faster; at 16 tokens, and for
//   W4A16 at 64, 3-6% slower, so those publish first like every other
//   contributor.)
// The acquire half of the arrival atomics, followed by a barrier, orders the
// finisher's reads after every other contributor's stores.  The finisher
// resets the counter for the next call.
constexpr int kSplitPublished = 1 << 16;   // above any arrival count (<= 1024 blocks)

struct PendingSplit {
  int64_t tile = -1;
  int old = 0;       // arrivals before this block's (thread 0 only)
  bool end = false;  // this block is the tile's first contributor, not yet arrived
};

template <int kCols, int kT>
__device__ __forceinline__ void split_publish(const KParams& p, int64_t tile, int64_t cta,
                                              int64_t nC, int64_t first_tile, int colbase, int r,
                                              int et, int epi_threads, const float* vals,
                                              PendingSplit& pend) {
  const int slot = (tile == first_tile) ? 0 : 1;
  float* mine = p.part + ((cta * 2 + slot) * kT) * kTileF;
#pragma unroll
  for (int c = 0; c < kCols; ++c) mine[(colbase + c) * kTileF + r] = vals[c];
  named_bar_sync(1, epi_threads);
  pend.tile = tile;
  pend.end = false;
  if (et == 0) pend.old = atomic_add_acq_rel_gpu(&p.counters[cta_of_step(tile * p.G, nC, p.W)], 1);
}

// Returns true when this block finishes the tile; `vals` then holds the
// tile's sum over all contributors in ascending block order.  For the tile's
// first contributor arriving late (kLate, pend.end) `vals` holds its own
// partial on entry.  Each
// other contributor's partial (T x 128 fp32, contiguous) comes into shared
// memory with one bulk copy, as many at a time as the idle weight and
// activation rings hold, so the sum costs one L2 round trip per batch
// instead of one per column chunk.
template <int kCols, int kT, bool kLate>
__device__ __forceinline__ bool split_finish(const KParams& p, Ctrl* ctrl, const PendingSplit& pend,
                                             int64_t cta, int64_t nC, int colbase, int r, int et,
                                             int epi_threads, float* vals, uint32_t stage_addr,
                                             const float* stage, uint32_t stage_bytes,
                                             uint32_t& fix_phase, const WaitCtx& ctx) {
  const int64_t G = p.G;
  const int64_t tile = pend.tile;
  const int64_t c_first = cta_of_step(tile * G, nC, p.W);
  const int64_t c_last = cta_of_step(tile * G + G - 1, nC, p.W);
  int* counter = &p.counters[c_first];
  const bool own = kLate && pend.end;   // this block is the first contributor, not yet arrived
  if (et == 0) {
    const int old = own ? atomic_add_acq_rel_gpu(counter, 1) : pend.old;
    ctrl->last_flag = ((old & (kSplitPublished - 1)) == static_cast<int>(c_last - c_first)) ? 1 : 0;
  }
  named_bar_sync(1, epi_threads);
  const bool last = ctrl->last_flag != 0;
  named_bar_sync(1, epi_threads);     // last_flag is rewritten below and by the next call
  if (!last) {
    if (own) {
      // another block finishes the tile: publish, then flag it
      float* mine = p.part + ((cta * 2 + 1) * kT) * kTileF;
#pragma unroll
      for (int c = 0; c < kCols; ++c) mine[(colbase + c) * kTileF + r] = vals[c];
      named_bar_sync(1, epi_threads);
      if (et == 0) red_add_release_gpu(counter, kSplitPublished);
    }
    return false;
  }
  // the first contributor's partial: in registers (pend.end), or published
  // after its arrival when its range started before the tile
  const bool first_late = kLate && !own && ((c_first * p.W / nC) / G != tile);
  if (first_late) {
    if (et == 0) {
      const uint64_t t0 = globaltimer_ns();
      int ok = 1;
      while ((ld_acquire_gpu(counter) & kSplitPublished) == 0) {
        if (globaltimer_ns() - t0 > ctx.limit_ns) {
          report_error(ctx.err, kDevTimeout, 21);
          ok = 0;
          break;
        }
      }
      ctrl->last_flag = ok;
    }
    named_bar_sync(1, epi_threads);
    const bool ok = ctrl->last_flag != 0;
    named_bar_sync(1, epi_threads);
    if (!ok) return false;
  }
  constexpr uint32_t kPartBytes = static_cast<uint32_t>(kT) * kTileF * sizeof(float);
  const int64_t cap = static_cast<int64_t>(stage_bytes / kPartBytes);
#pragma unroll
  for (int c = 0; c < kCols; ++c) vals[c] = own ? 0.0f + vals[c] : 0.0f;
  const int64_t from = own ? c_first + 1 : c_first;
  bool ok = true;
  for (int64_t b0 = from; b0 <= c_last; b0 += cap) {
    const int64_t nb = (c_last - b0 + 1) < cap ? (c_last - b0 + 1) : cap;
    if (et == 0) {
      // the rings were last touched by generic loads and stores (converters,
      // the previous batch's sums), and the partials were written by other
      // blocks' generic stores (acquired through the arrival counter): order
      // both before the async copies
      fence_proxy_async_smem();
      fence_proxy_async_global();
      const uint32_t full = smem_u32(&ctrl->fix_full);
      mbar_arrive_expect_tx(full, static_cast<uint32_t>(nb) * kPartBytes);
      for (int64_t i = 0; i < nb; ++i) {
        const int64_t cc = b0 + i;
        const int slot = ((cc * p.W / nC) / G == tile) ? 0 : 1;
        bulk_load(stage_addr + static_cast<uint32_t>(i) * kPartBytes,
                  p.part + ((cc * 2 + slot) * kT) * kTileF, kPartBytes, full);
      }
    }
    ok = warp_all(mbar_wait(smem_u32(&ctrl->fix_full), fix_phase, ctx, 18));
    fix_phase ^= 1u;
    if (ok) {
      for (int64_t i = 0; i < nb; ++i) {
        const float* src = stage + i * (kPartBytes / sizeof(float)) + colbase * kTileF + r;
#pragma unroll
        for (int c = 0; c < kCols; ++c) vals[c] += src[c * kTileF];
      }
    }
    named_bar_sync(1, epi_threads);   // the next batch overwrites the staging area
    if (!ok) return false;
  }
  if (et == 0) *counter = 0;
  return true;
}

template <int kMode, int T, int GPS>
__global__ void __launch_bounds__(Cfg<kMode, T, GPS>::kThreads, 1)
    qlin_gemm_kernel(const __grid_constant__ CUtensorMap tm_w,
                     const __grid_constant__ CUtensorMap tm_a,
                     const __grid_constant__ CUtensorMap tm_s, const KParams p) {
  using C = Cfg<kMode, T, GPS>;
  constexpr int NB = C::kNumBuf;
  constexpr int ND = C::kWO ? C::kSegBufs : C::kNumD;
  constexpr int SR = C::kScaleSlots;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const int stages = p.stages;
  constexpr int NX = C::kXSlots;                 // 16-bit operand slots
  constexpr int NXR = C::kXConv ? C::kXiSlots : C::kXSlots;   // slots the producer fills
  const uint32_t x_off = static_cast<uint32_t>(stages) * C::kStageBytes;
  const uint32_t xi_off = x_off + static_cast<uint32_t>(NX) * C::kABytes;
  const uint32_t sc_off = xi_off + static_cast<uint32_t>(C::kXiSlots) * C::kXiBytes;
  const uint16_t* scale_ring = reinterpret_cast<const uint16_t*>(smem + sc_off);
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(smem + sc_off + C::kScaleBytes);
  unsigned long long* skeys =
      reinterpret_cast<unsigned long long*>(smem + sc_off + C::kScaleBytes + kCtrlBytes);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t nC = gridDim.x;
  const int64_t cta = blockIdx.x;
  // stream-K: the block's range [s0, s1) of the step list; banded tiles: the
  // block's whole tiles cta, cta + nC, ... (s0 unused)
  const int64_t s0 = p.band > 0 ? 0 : cta * p.W / nC;
  const int64_t s1 = p.band > 0 ? 0 : (cta + 1) * p.W / nC;
  const int n_steps = p.band > 0
                          ? static_cast<int>(((p.TT * p.F - cta + nC - 1) / nC) * p.G)
                          : static_cast<int>(s1 - s0);
  const int64_t G = p.G;
  const int64_t F = p.F;
  // weights: streamed once (stream-K), or shared by the blocks of a band that
  // read each tile within microseconds of each other (banded tiles)
  const uint64_t pol_w = p.band > 0 ? policy_evict_normal() : policy_evict_first();
  const uint64_t pol_a = policy_evict_last();
  int w_issued = 0;   // weight loads issued by the weight producer (warp 0, lane 0)

  if (threadIdx.x == 0) {
    for (int i = 0; i < stages; ++i) {
      mbar_init(smem_u32(&ctrl->wfull[i]), 1);
      mbar_init(smem_u32(&ctrl->empty[i]), C::kEmptyCount);
    }
    for (int i = 0; i < NXR; ++i) {
      mbar_init(smem_u32(&ctrl->xfull[i]), 1);
      mbar_init(smem_u32(&ctrl->xempty[i]), C::kXConv ? C::kConvWarps / 2 : 1);
    }
    for (int i = 0; i < NB; ++i) {
      mbar_init(smem_u32(&ctrl->a_full[i]), C::kConvWarps / 2);
      mbar_init(smem_u32(&ctrl->a_empty[i]), 1);
    }
    for (int i = 0; i < ND; ++i) {
      mbar_init(smem_u32(&ctrl->d_full[i]), C::kWO ? C::kIssuers : 1);
      mbar_init(smem_u32(&ctrl->d_empty[i]), C::kEpiWarps);
    }
    for (int i = 0; i < SR; ++i) {
      mbar_init(smem_u32(&ctrl->s_full[i]), 1);
      // released by every converter warp (weight-only) or epilogue warp (W8A8)
      mbar_init(smem_u32(&ctrl->s_empty[i]), C::kWO ? C::kConvWarps : C::kEpiWarps);
    }
    mbar_init(smem_u32(&ctrl->mma_done), C::kIssuers);
    mbar_init(smem_u32(&ctrl->x_go), 1);
    mbar_init(smem_u32(&ctrl->fix_full), 1);
    ctrl->abort_flag = 0;
    ctrl->last_flag = 0;
    fence_barrier_init();
    // The weights depend on nothing: start streaming them before the block's
    // set-up barrier (every slot is free, so no wait is needed).  Only a few:
    // every TMA load of the SM queues behind the ones issued before it, and
    // the first activation tiles must not wait behind a full weight ring.
    if (p.wtiles == nullptr) prefetch_tmap(&tm_w);
    StepIter it(p, s0);
    const int pre = kPreW < stages ? kPreW : stages;
    const int first = n_steps < pre ? n_steps : pre;
    for (int j = 0; j < first; ++j, it.next()) {
      const uint32_t full = smem_u32(&ctrl->wfull[j]);
      mbar_arrive_expect_tx(full, C::kWBytes);
      load_weights<C>(sbase + static_cast<uint32_t>(j) * C::kStageBytes, &tm_w, p, it, full, pol_w);
    }
    w_issued = first;
  }
  __syncwarp();
  if (warp == 1) {
    tmem_alloc(smem_u32(&ctrl->tmem_base), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  grid_dep_launch();
  const uint32_t tmem = ctrl->tmem_base;
  const WaitCtx ctx{p.err, &ctrl->abort_flag, p.limit_ns};
  int never_abort = 0;
  const WaitCtx drain_ctx{p.err, &never_abort, p.limit_ns};

  if (warp == 0) {
    // ------------------------------------------------------ weight producer
    if (lane == 0) {
      StepIter it(p, s0);
      Ring rg(stages);
      for (int j = 0; j < w_issued; ++j) {
        it.next();
        rg.next();
      }
      const int first_w = w_issued;
      for (int j = w_issued; j < n_steps; ++j, it.next(), rg.next()) {
        // The weight-only formats read bf16 activations that are usually
        // ready at launch, so their first tiles go ahead of the weight ring
        // (x_go).  W8A8 activations come from the act-quant kernel launched
        // just before: the weights fill the ring while it runs.
        if (C::kWO && j == first_w && !mbar_wait(smem_u32(&ctrl->x_go), 0u, ctx, 19)) break;
        if (!mbar_wait(smem_u32(&ctrl->empty[rg.slot]), rg.phase ^ 1u, ctx, 1)) break;
        const uint32_t full = smem_u32(&ctrl->wfull[rg.slot]);
        mbar_arrive_expect_tx(full, C::kWBytes);
        load_weights<C>(sbase + static_cast<uint32_t>(rg.slot) * C::kStageBytes, &tm_w, p, it, full,
                        pol_w);
        ++w_issued;
      }
      // Every load issued must land before the block exits.
      for (int j = w_issued > stages ? w_issued - stages : 0; j < w_issued; ++j)
        (void)mbar_wait(smem_u32(&ctrl->wfull[j % stages]),
                        static_cast<uint32_t>(j / stages) & 1u, drain_ctx, 2);
    }
    __syncwarp();
  } else if (warp == 2) {
    // ------------------------------------ activation and scale producer
    if (lane == 0) {
      prefetch_tmap(&tm_a);
      if constexpr (C::kScales) prefetch_tmap(&tm_s);
      StepIter it(p, s0);
      Ring rg(NXR);
      ChunkIter ch;
      int issued = 0, s_issued = 0;
      bool waited = false;
      const int x_first = n_steps < NXR ? n_steps : NXR;   // loads before the weights resume
      bool go = false;
      for (int j = 0; j < n_steps; ++j, it.next(), rg.next(), ch.advance()) {
        if constexpr (C::kScales) {
          if (ch.begin(j == 0 || it.g == 0)) {
            const int slot = ch.ci % SR;
            const uint32_t sph = static_cast<uint32_t>(ch.ci / SR) & 1u;
            // Short segments can fill the scale ring before the first
            // activation tiles are all issued; the ring drains only as the
            // weights flow, so release the weight producer before waiting.
            if (!go && ch.ci >= SR) {
              mbar_arrive(smem_u32(&ctrl->x_go));
              go = true;
            }
            if (!mbar_wait(smem_u32(&ctrl->s_empty[slot]), sph ^ 1u, ctx, 11)) break;
            const uint32_t sfull = smem_u32(&ctrl->s_full[slot]);
            mbar_arrive_expect_tx(sfull, p.s_tx);
            const int32_t srow = kMode == kModeW8A16 ? static_cast<int32_t>(it.g * p.s_rps)
                                                     : static_cast<int32_t>(it.g * GPS);
            tma_load_2d(sbase + sc_off + static_cast<uint32_t>(slot) * C::kScaleSlotBytes, &tm_s,
                        sfull, static_cast<int32_t>(it.f * kTileF), srow, pol_w);
            ++s_issued;
          }
        }
        if (!mbar_wait(smem_u32(&ctrl->xempty[rg.slot]), rg.phase ^ 1u, ctx, 15)) break;
        if (!waited) {
          grid_dep_wait();   // the activations come from the previous kernel
          waited = true;
        }
        const uint32_t full = smem_u32(&ctrl->xfull[rg.slot]);
        if constexpr (!C::kXConv) {
          const uint32_t dst = sbase + x_off + static_cast<uint32_t>(rg.slot) * C::kABytes;
          mbar_arrive_expect_tx(full, C::kABytes);
          // one load brings both 64-wide halves of the group, each as a T x
          // 128 B swizzled tile (the activations seen as [K/64][M][64])
          tma_load_3d(dst, &tm_a, full, 0, static_cast<int32_t>(it.t * T),
                      static_cast<int32_t>(it.g * 2 * GPS), pol_a);
        } else {
          // the group's int8 tile, T rows x 128 B, 128-byte swizzled
          const uint32_t dst = sbase + xi_off + static_cast<uint32_t>(rg.slot) * C::kXiBytes;
          mbar_arrive_expect_tx(full, C::kXiBytes);
          tma_load_2d(dst, &tm_a, full, static_cast<int32_t>(it.g * kGroup),
                      static_cast<int32_t>(it.t * T), pol_a);
        }
        ++issued;
        if (!go && issued == x_first) {
          mbar_arrive(smem_u32(&ctrl->x_go));
          go = true;
        }
      }
      if (!go) mbar_arrive(smem_u32(&ctrl->x_go));
      for (int j = issued > NXR ? issued - NXR : 0; j < issued; ++j)
        (void)mbar_wait(smem_u32(&ctrl->xfull[j % NXR]), static_cast<uint32_t>(j / NXR) & 1u,
                        drain_ctx, 16);
      for (int c = s_issued > SR ? s_issued - SR : 0; c < s_issued; ++c)
        (void)mbar_wait(smem_u32(&ctrl->s_full[c % SR]), static_cast<uint32_t>(c / SR) & 1u,
                        drain_ctx, 12);
    }
    __syncwarp();
  } else if (warp == 1 || warp == 3) {
    // ----------------------------------------------------------- MMA issuers
    // warp 1 takes the even steps, warp 3 the odd ones
    if (lane == 0) {
      const int me = warp == 1 ? 0 : 1;
      constexpr uint32_t idesc = idesc_f16(kTileF, T, C::kWO);
      StepIter it(p, s0);
      Ring rx(NX);
      int seg = 0;
      bool started = false;   // W4A16: this issuer has accumulated into the segment
      for (int j = 0; j < n_steps; ++j, it.next(), rx.next()) {
        const bool seg_first = (j == 0) || (it.g == 0);
        const bool seg_last = (j == n_steps - 1) || (it.g == G - 1);
        const int ab = j % NB;
        const uint32_t abph = static_cast<uint32_t>(j / NB) & 1u;
        if (seg_first) started = false;
        const int didx = C::kWO ? seg : j;
        const int db = didx % ND;
        const uint32_t dbph = static_cast<uint32_t>(didx / ND) & 1u;
        const uint32_t dcol = C::kWO ? tmem + C::kColD + (db * C::kIssuers + me) * T
                                     : tmem + C::kColD + db * T;
        if ((j & 1) == me) {
          const bool need_d = C::kWO ? !started : true;
          // in-kernel expansion: a_full also covers the fp16 operand slot
          // (slot ab, written by the same converter group); else the TMA tile
          if (!C::kXConv && !mbar_wait(smem_u32(&ctrl->xfull[rx.slot]), rx.phase, ctx, 3)) break;
          if (!mbar_wait(smem_u32(&ctrl->a_full[ab]), abph, ctx, 4)) break;
          if (need_d && !mbar_wait(smem_u32(&ctrl->d_empty[db]), dbph ^ 1u, ctx, 5)) break;
          tc_fence_after();
          const uint32_t xb = sbase + x_off + static_cast<uint32_t>(rx.slot) * C::kABytes;
          const uint64_t d0 = smem_desc(xb, 16u, 1024u, 2u);
#pragma unroll
          for (int ks = 0; ks < 8 * GPS; ++ks) {
            // 128-byte swizzled K-major 16-bit tile: 8-row groups 1024 B
            // apart, K advanced by 32 B (16 elements) inside the 128-byte row;
            // the second 64-wide half of the group starts T*128 B further.
            const uint32_t off = static_cast<uint32_t>(ks >> 2) * (T * 128u) +
                                 static_cast<uint32_t>(ks & 3) * 32u;
            const bool acc = C::kWO ? (started || ks > 0) : ks > 0;
            mma_ts(dcol, tmem + C::kColA + ab * C::kACols + ks * 8, d0 + (off >> 4), idesc,
                   acc ? 1u : 0u);
          }
          if constexpr (C::kACommit) tc_commit(smem_u32(&ctrl->a_empty[ab]));
          if constexpr (!C::kXConv) tc_commit(smem_u32(&ctrl->xempty[rx.slot]));
          // W8A8: also frees the A buffer (and the fp16 slot of in-kernel expansion)
          if constexpr (!C::kWO) tc_commit(smem_u32(&ctrl->d_full[db]));
          started = true;
        }
        if constexpr (C::kWO) {
          if (seg_last) {
            // Every issuer reports on every segment.  One that accumulated
            // nothing into it arrives directly, but only once the epilogue has
            // released this buffer's previous segment, so that its arrival
            // cannot complete that earlier phase in the other issuer's place.
            if (started) {
              tc_commit(smem_u32(&ctrl->d_full[db]));
            } else {
              if (!mbar_wait(smem_u32(&ctrl->d_empty[db]), dbph ^ 1u, ctx, 17)) break;
              mbar_arrive(smem_u32(&ctrl->d_full[db]));
            }
            ++seg;
          }
        }
      }
      tc_commit(smem_u32(&ctrl->mma_done));
      (void)mbar_wait(smem_u32(&ctrl->mma_done), 0u, drain_ctx, 6);
    }
    __syncwarp();
  } else if (warp >= C::kConvWarp0 && warp < C::kEpiWarp0) {
    // ------------------------------------------------------------ converters
    // group 0 (warps 4-7) takes the even steps, group 1 (warps 8-11) the odd
    // ones, so one group's load/convert/store latency overlaps the other's
    const int ct = threadIdx.x - 32 * C::kConvWarp0;      // 0..255
    const int grp = ct >> 7;
    const int r = ct & 127;                                // row of A = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    StepIter it(p, s0);
    Ring rg(stages);
    Ring ri(C::kXConv ? NXR : 1);   // in-kernel expansion: int8 staging slot of the step
    ChunkIter ch;
    bool chunk_ready = false;   // W4A16: this group has waited for the chunk's scales
    for (int j = 0; j < n_steps; ++j, it.next(), rg.next(), ri.next(), ch.advance()) {
      const bool seg_last = (j == n_steps - 1) || (it.g == G - 1);
      if constexpr (C::kWO) {
        if (ch.begin(j == 0 || it.g == 0)) chunk_ready = false;
      }
      const bool mine = (j & 1) == grp;
      if (mine) {
        const int ab = j % NB;
        const uint32_t abph = static_cast<uint32_t>(j / NB) & 1u;
        if (!warp_all(mbar_wait(smem_u32(&ctrl->wfull[rg.slot]), rg.phase, ctx, 7))) break;
        // Every word this thread converts in the step, loaded before it waits
        // for its A buffer (and before the first TMEM store, whose ordering
        // would otherwise hold each batch of shared-memory loads back behind
        // the previous batch's conversion); the weight slot is then free for
        // the next load.
        const uint32_t* wsm = reinterpret_cast<const uint32_t*>(
            smem + static_cast<uint32_t>(rg.slot) * C::kStageBytes);
        uint32_t wreg[C::kWordRows];
#pragma unroll
        for (int i = 0; i < C::kWordRows; ++i) wreg[i] = wsm[i * kTileF + r];
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctrl->empty[rg.slot]));
        bool ok = true;
        if constexpr (C::kACommit) {
          if (ok) ok = mbar_wait(smem_u32(&ctrl->a_empty[ab]), abph ^ 1u, ctx, 8);
        } else if (ok && j >= NB) {
          // A buffer ab was last read by step j - NB, committed on its D
          // buffer.  That buffer's next completion is step j - NB + ND, which
          // (ND - NB even) belongs to this converter group and so comes after
          // this conversion: the parity below cannot be overtaken.
          const int pj = j - NB;
          ok = mbar_wait(smem_u32(&ctrl->d_full[pj % ND]), static_cast<uint32_t>(pj / ND) & 1u,
                         ctx, 8);
        }
        if (C::kXConv && ok) ok = mbar_wait(smem_u32(&ctrl->xfull[ri.slot]), ri.phase, ctx, 3);
        uint32_t s2g[GPS];                     // W4A16: bf16x2 scale of each group of the step
#pragma unroll
        for (int gi = 0; gi < GPS; ++gi) s2g[gi] = 0u;
        float sq[4] = {0.f, 0.f, 0.f, 0.f};   // W8A16 scales of the group's quarters
        if constexpr (C::kWO) {
          const int slot = ch.ci % SR;
          if (ok && !chunk_ready)
            ok = mbar_wait(smem_u32(&ctrl->s_full[slot]), static_cast<uint32_t>(ch.ci / SR) & 1u,
                           ctx, 13);
          if (!warp_all(ok)) break;
          chunk_ready = true;
          if constexpr (C::kInt4) {
#pragma unroll
            for (int gi = 0; gi < GPS; ++gi) {
              const uint32_t sb = scale_ring[(slot * C::kScaleRowsMax + ch.row() * GPS + gi) * 128 + r];
              s2g[gi] = sb | (sb << 16);
            }
          } else {
            // W8A16: the scale of each 32-wide quarter of the group
            const uint16_t* srow = scale_ring + (slot * C::kScaleRowsMax + ch.row() * p.s_rps) * 128 + r;
#pragma unroll
            for (int h = 0; h < 4; ++h)
              sq[h] = __uint_as_float(static_cast<uint32_t>(srow[(p.s_rps == 4 ? h : 0) * 128]) << 16);
          }
        } else {
          if (!warp_all(ok)) break;
        }
        tc_fence_after();
        if constexpr (C::kXConv) {
          // The step's int8 tokens (T rows x 128, 128-byte swizzled) become
          // the fp16 B operand in slot ab: two 64-wide halves of T rows x
          // 128 B, 128-byte swizzled.  q + 128 as a biased byte -> exact fp16.
          const uint8_t* xi = smem + xi_off + static_cast<uint32_t>(ri.slot) * C::kXiBytes;
          uint8_t* xf = smem + x_off + static_cast<uint32_t>(ab) * C::kABytes;
#pragma unroll
          for (int q = r; q < 8 * T; q += kTileF) {
            const int row = q >> 3;      // token row of the tile
            const int c = q & 7;         // 16-byte chunk = 16 K values
            const uint4 raw = *reinterpret_cast<const uint4*>(xi + row * 128 + ((c ^ (row & 7)) << 4));
            uint4 o0, o1;
            biased_u8x4_to_f16x4(raw.x ^ 0x80808080u, o0.x, o0.y);
            biased_u8x4_to_f16x4(raw.y ^ 0x80808080u, o0.z, o0.w);
            biased_u8x4_to_f16x4(raw.z ^ 0x80808080u, o1.x, o1.y);
            biased_u8x4_to_f16x4(raw.w ^ 0x80808080u, o1.z, o1.w);
            uint8_t* dst = xf + (c >> 2) * (T * 128) + row * 128;
            const int c2 = (c & 3) * 2;
            *reinterpret_cast<uint4*>(dst + ((c2 ^ (row & 7)) << 4)) = o0;
            *reinterpret_cast<uint4*>(dst + (((c2 + 1) ^ (row & 7)) << 4)) = o1;
          }
          fence_proxy_async_smem();   // generic writes -> the MMA's async reads
        }
        const uint32_t acol = tmem + lane_off + C::kColA + ab * C::kACols;
#pragma unroll
        for (int h = 0; h < 4 * GPS; ++h) {
          uint32_t v[16];
          if constexpr (C::kInt4) {
#pragma unroll
            for (int i = 0; i < 4; ++i) int4x8_to_bf16x8(wreg[h * 4 + i], s2g[h >> 2], v + 4 * i);
          } else if constexpr (kMode == kModeW8A16) {
            // byte u = q + 128 -> exact q in fp32 (2^23 + u minus 2^23 + 128),
            // q * s exact in fp32, one rounding to bf16
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const uint32_t w = wreg[h * 8 + i];
              float f[4];
#pragma unroll
              for (int b = 0; b < 4; ++b)
                f[b] = (__uint_as_float(prmt(w, 0x4B000000u, static_cast<uint32_t>(b | 0x7440))) -
                        8388736.0f) * sq[h];
              v[2 * i] = bf16x2_rn(f[0], f[1]);
              v[2 * i + 1] = bf16x2_rn(f[2], f[3]);
            }
          } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) biased_u8x4_to_f16x4(wreg[h * 8 + i], v[2 * i], v[2 * i + 1]);
          }
          tmem_st16(acol + h * 16, v);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if constexpr (C::kXConv) mbar_arrive(smem_u32(&ctrl->xempty[ri.slot]));
          mbar_arrive(smem_u32(&ctrl->a_full[ab]));
        }
      }
      if constexpr (C::kWO) {
        // Both groups release each scale chunk.  A group that had no step in
        // the chunk read nothing from it, but it still waits for the chunk to
        // land first: with one-step chunks (tiles of one K group) a group
        // could otherwise run several chunks ahead, complete an earlier
        // chunk's release phase in the other group's place, and let the
        // producer reload a slot that the other group still reads.
        if (ch.ends(seg_last)) {
          if (!chunk_ready &&
              !warp_all(mbar_wait(smem_u32(&ctrl->s_full[ch.ci % SR]),
                                  static_cast<uint32_t>(ch.ci / SR) & 1u, ctx, 20)))
            break;
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&ctrl->s_empty[ch.ci % SR]));
        }
      }
    }
    __syncwarp();
  } else if (warp >= C::kEpiWarp0) {
    // ------------------------------------------------------------ epilogue
    const int et = threadIdx.x - 32 * C::kEpiWarp0;        // 0..255
    const int r = (warp & 3) * 32 + lane;                  // TMEM lane = feature in tile
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int colbase = ((warp - C::kEpiWarp0) >> 2) * C::kEpiCols;
    const int64_t M = p.M, N = p.N;
    const int64_t first_tile = s0 / G;
    uint16_t* y = static_cast<uint16_t*>(p.out);
    float acc[C::kEpiCols];
    bool alive = true;          // false once this warp's waits gave up
    int64_t seg_g0 = 0;
    int seg = 0;
    int seg_j0 = 0;             // first step of the current segment
    bool waited = false;
    PendingSplit pend[2];       // at most the first and the last tile of the range
    int npend = 0;
    unsigned long long run_key[2] = {0ull, 0ull};   // greedy argmax: tokens lane, lane + 32
    // Every final output value passes through here exactly once (full tiles
    // at their segment end, split tiles in the last contributor).  All
    // threads of each warp call it together.
    auto write_out = [&](int64_t tt, int64_t nn, const float* vals) {
      if (p.amax_keys) {
        // greedy argmax: key = order-preserving bits of the bf16 value << 32
        // | ~n, so the largest key is the largest value at the lowest n; the
        // warp's 32 features reduce by shuffles, the block's in shared memory
        // The warp's 32 lanes hold 32 consecutive columns (nn - lane + 0..31),
        // so within the warp a 32-bit key (value bits << 16 | 31 - lane)
        // finds the same winner with one redux; lane 0 then forms the 64-bit
        // key with the winning column.
        if (tt * T + colbase >= M) return;            // no valid token in this half
        const int64_t n0 = nn - lane;                  // column of lane 0
#pragma unroll
        for (int c = 0; c < C::kEpiCols; ++c) {
          const int64_t m = tt * T + colbase + c;
          uint32_t key = 0u;
          if (nn < N && m < M) {
            const float v = C::kWO ? vals[c] : vals[c] * __ldg(p.s_a + m);
            uint32_t b = __bfloat16_as_ushort(__float2bfloat16_rn(v));
            if (b == 0x8000u) b = 0u;   // -0 equals +0
            const uint32_t ord = (b & 0x8000u) ? (~b & 0xFFFFu) : (b | 0x8000u);
            key = (ord << 16) | static_cast<uint32_t>(31 - lane);
          }
          const uint32_t best = __reduce_max_sync(0xFFFFFFFFu, key);
          if (best != 0u && lane == (c & 31)) {
            // token c's running best lives in lane c % 32 of this warp
            const uint32_t n_win = static_cast<uint32_t>(n0 + (31 - static_cast<int>(best & 0xFFFFu)));
            const unsigned long long k64 = (static_cast<unsigned long long>(best >> 16) << 32) |
                                           static_cast<unsigned long long>(~n_win);
            if (k64 > run_key[c >> 5]) run_key[c >> 5] = k64;
          }
        }
        return;
      }
      if (nn >= N) return;
#pragma unroll
      for (int c = 0; c < C::kEpiCols; ++c) {
        const int64_t m = tt * T + colbase + c;
        if (m < M) {
          const float v = C::kWO ? vals[c] : vals[c] * __ldg(p.s_a + m);
          y[m * N + nn] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
        }
      }
    };
    StepIter it(p, s0);
    ChunkIter ch;
    for (int j = 0; j < n_steps; ++j, it.next(), ch.advance()) {
      const int64_t g = it.g, t = it.t;
      const int64_t n = it.f * kTileF + r;
      const bool seg_first = (j == 0) || (g == 0);
      const bool seg_last = (j == n_steps - 1) || (g == G - 1);
      if (seg_first) {
        seg_g0 = g;
        seg_j0 = j;
#pragma unroll
        for (int c = 0; c < C::kEpiCols; ++c) acc[c] = 0.0f;
      }
      if (!C::kWO || seg_last) {
        // drain one accumulator buffer: per group (W8A8) or per segment (W4A16)
        const int idx = C::kWO ? seg : j;
        const int b = idx % ND;
        const uint32_t bph = static_cast<uint32_t>(idx / ND) & 1u;
        float sw = 0.0f;
        if constexpr (kMode == kModeW8A8) {
          ch.begin(seg_first);
          const int slot = ch.ci % SR;
          if (alive && ch.row() == 0)
            alive = warp_all(mbar_wait(smem_u32(&ctrl->s_full[slot]),
                                       static_cast<uint32_t>(ch.ci / SR) & 1u, ctx, 14));
          if (alive) {
            sw = __half2float(__ushort_as_half(scale_ring[(slot * kScaleChunk + ch.row()) * 128 + r]));
            if (ch.ends(seg_last)) {
              __syncwarp();
              if (lane == 0) mbar_arrive(smem_u32(&ctrl->s_empty[slot]));
            }
          }
        }
        if (alive) alive = warp_all(mbar_wait(smem_u32(&ctrl->d_full[b]), bph, ctx, 9));
        if (alive) {
          tc_fence_after();
          const uint32_t dcol = tmem + lane_off + C::kColD + colbase +
                                (C::kWO ? b * C::kIssuers * T : b * T);
          constexpr int E = C::kEpiCols;
          uint32_t v[E];
          if constexpr (C::kWO) {
            // the issuers' accumulators, summed in issuer order; an issuer
            // that took no step of this segment left its accumulator unused
            const bool both = j > seg_j0;
            const int only = seg_j0 & 1;
            if (both) {
              tmem_ld_cols<E>(dcol, v);
              tmem_ld_cols<E>(dcol + T, reinterpret_cast<uint32_t*>(acc));
              tmem_wait_ld();
#pragma unroll
              for (int c = 0; c < E; ++c) acc[c] = __uint_as_float(v[c]) + acc[c];
            } else {
              tmem_ld_cols<E>(dcol + (only == 0 ? 0u : static_cast<uint32_t>(T)),
                              reinterpret_cast<uint32_t*>(acc));
              tmem_wait_ld();
            }
          } else {
            // all of this thread's columns in one batch of loads, one wait
            tmem_ld_cols<E>(dcol, v);
            tmem_wait_ld();
            if constexpr (kMode == kModeP) {
              if (!waited) {
                grid_dep_wait();
                waited = true;
              }
              int32_t* P = static_cast<int32_t*>(p.out);
#pragma unroll
              for (int c = 0; c < E; ++c) {
                const int64_t m = t * T + colbase + c;
                if (m < M && n < N)
                  P[(g * M + m) * N + n] = static_cast<int32_t>(__uint_as_float(v[c]));
              }
            } else {
#pragma unroll
              for (int c = 0; c < E; ++c) acc[c] = fmaf(__uint_as_float(v[c]), sw, acc[c]);
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&ctrl->d_empty[b]));
        }
      }
      if (C::kWO && seg_last) ++seg;
      if (kMode == kModeP || !seg_last) continue;

      // ---- end of this block's segment of the tile (all epilogue warps agree)
      if (!named_bar_and(2, C::kEpiThreads, alive)) break;
      if (!waited) {
        grid_dep_wait();   // outputs and workspace may still be in use upstream
        waited = true;
      }
      const int64_t tile = it.tile();
      const bool full_tile = (seg_g0 == 0) && (g == G - 1);
      if (full_tile) {
        write_out(t, n, acc);
      } else if (!C::kWO && T >= 64 && tile != first_tile) {
        // the range ends inside this tile (its last segment): this block is
        // the tile's first contributor and arrives after the loop, with its
        // partial still in acc
        pend[npend].tile = tile;
        pend[npend].end = true;
        ++npend;
      } else {
        split_publish<C::kEpiCols, T>(p, tile, cta, nC, first_tile, colbase, r, et, C::kEpiThreads,
                                   acc, pend[npend]);
        ++npend;
      }
    }
    // the split tiles this block took part in: the last block to arrive sums
    // the partials and writes the output
    if (named_bar_and(2, C::kEpiThreads, alive)) {
      uint32_t fix_phase = 0;
      // the last tile first: its partial is still in acc
      for (int k = npend - 1; k >= 0; --k) {
        if (split_finish<C::kEpiCols, T, (!C::kWO && T >= 64)>(p, ctrl, pend[k], cta, nC, colbase, r, et,
                                                  C::kEpiThreads,
                                      acc, sbase, reinterpret_cast<const float*>(smem), sc_off,
                                      fix_phase, drain_ctx)) {
          const int64_t tt = pend[k].tile / F;
          write_out(tt, (pend[k].tile - tt * F) * kTileF + r, acc);
        }
      }
      if (p.amax_keys) {
        // the block's best column per token (one token tile: M <= T): the
        // four lane-quarter warps of each column half meet in shared memory
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int c = lane + 32 * i;
          if (c < C::kEpiCols) skeys[(warp & 3) * kTileF + colbase + c] = run_key[i];
        }
        named_bar_sync(1, C::kEpiThreads);
        if (et < T && et < M) {
          unsigned long long k = skeys[et];
#pragma unroll
          for (int q = 1; q < 4; ++q) k = skeys[q * kTileF + et] > k ? skeys[q * kTileF + et] : k;
          if (k != 0ull) {
            if (!waited) grid_dep_wait();
            atomicMax(&p.amax_keys[et], k);
          }
        }
      }
    }
    __syncwarp();
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// int8 activations -> fp16 (exact), 16 values per thread: the B operand of
// the W8A8 GEMM at token tiles of 64 and more.  Waits for its predecessor
// before touching memory (the previous GEMM may still read this buffer), then
// lets the GEMM start.
__global__ void __launch_bounds__(256) act_i8_to_f16_kernel(const int8_t* __restrict__ q,
                                                            uint16_t* __restrict__ out,
                                                            int64_t n16) {
  grid_dep_wait();
  grid_dep_launch();
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n16;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint4 raw = __ldg(reinterpret_cast<const uint4*>(q) + i);
    uint4 o0, o1;
    biased_u8x4_to_f16x4(raw.x ^ 0x80808080u, o0.x, o0.y);
    biased_u8x4_to_f16x4(raw.y ^ 0x80808080u, o0.z, o0.w);
    biased_u8x4_to_f16x4(raw.z ^ 0x80808080u, o1.x, o1.y);
    biased_u8x4_to_f16x4(raw.w ^ 0x80808080u, o1.z, o1.w);
    reinterpret_cast<uint4*>(out)[2 * i] = o0;
    reinterpret_cast<uint4*>(out)[2 * i + 1] = o1;
  }
}

// fp16 codes -> int8 codes (exact: the values are integers in [-127, 127]),
// 8 per thread: the int8 input of the W8A8 GEMM at token tiles of 32 and
// fewer, which expand int8 tiles themselves.  Ordered like the kernel above.
__global__ void __launch_bounds__(256) act_f16_to_i8_kernel(const uint16_t* __restrict__ c,
                                                            int8_t* __restrict__ out,
                                                            int64_t n8) {
  grid_dep_wait();
  grid_dep_launch();
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n8;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint4 h = __ldg(reinterpret_cast<const uint4*>(c) + i);
    const uint32_t w[4] = {h.x, h.y, h.z, h.w};
    uint32_t b[2] = {0u, 0u};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint16_t bits = static_cast<uint16_t>(w[j >> 1] >> (16 * (j & 1)));
      const int v = __half2int_rn(__ushort_as_half(bits));
      b[j >> 2] |= (static_cast<uint32_t>(v) & 0xFFu) << (8 * (j & 3));
    }
    reinterpret_cast<uint2*>(out)[i] = make_uint2(b[0], b[1]);
  }
}

// Greedy argmax: the column index encoded in each row's key.
__global__ void __launch_bounds__(128) argmax_finalize_kernel(const unsigned long long* keys,
                                                              int64_t M, int32_t* idx) {
  grid_dep_wait();
  grid_dep_launch();
  const int64_t m = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  if (m < M) {
    const unsigned long long k = keys[m];
    idx[m] = k ? static_cast<int32_t>(~static_cast<uint32_t>(k & 0xFFFFFFFFull)) : -1;
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

// 16-bit activations [M][K] seen as a 3D tensor {64 (k inside a half group),
// M (rows, stride K*2 bytes), K/64 (half groups, stride 128 bytes)}; a box
// {64, T, 2g} is g 128-wide K groups as 2g swizzled T x 128 B tiles.
bool make_act_map(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t M,
                  uint64_t K, uint32_t T, uint32_t halves) {
  EncodeFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {64, M, K / 64};
  const cuuint64_t strides[2] = {K * 2, 128};
  const cuuint32_t box[3] = {64, T, halves};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, dtype, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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

}  // namespace

namespace {

template <int kMode, int T, int GPS>
cudaError_t launch_t(const GemmArgs& a, const GemmPlan& pl_in, int* err, cudaStream_t stream) {
  using C = Cfg<kMode, T, GPS>;
  // steps of GPS groups: fewer (tile, step) units, never more blocks; the
  // minimum work per block stays kMinSteps groups
  GemmPlan pl = pl_in;
  if (GPS > 1) {
    pl.G = pl_in.G / GPS;
    pl.steps = pl.TT * pl.F * pl.G;
    if (pl.band == 0) {
      const int64_t by_work = (pl.steps * GPS + kMinSteps - 1) / kMinSteps;
      pl.ctas = by_work < pl_in.ctas ? by_work : pl_in.ctas;
      if (pl.ctas < 1) pl.ctas = 1;
    }
  }
  const void* act16 = a.act;   // 16-bit activation tiles (TMA)
  const void* act8 = a.act;    // int8 activation tiles (in-kernel expansion)
  if constexpr (C::kXConv) {
    if (a.act_c16) {
      // fp16 codes -> int8 codes in the workspace
      int8_t* dst = static_cast<int8_t*>(a.workspace) + pl.act_offset;
      const int64_t n8 = a.M * a.K / 8;
      int64_t blocks = (n8 + 255) / 256;
      if (blocks > 4096) blocks = 4096;
      cudaError_t e = launch_pdl(act_f16_to_i8_kernel, dim3(static_cast<unsigned>(blocks)),
                                 dim3(256), 0, stream, static_cast<const uint16_t*>(a.act), dst, n8);
      if (e != cudaSuccess) return e;
      act8 = dst;
    }
  }
  if constexpr (!C::kWO && !C::kXConv) {
    if (!a.act_c16) {
      // int8 codes -> fp16 image in the workspace
      uint16_t* dst =
          reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(a.workspace) + pl.act_offset);
      const int64_t n16 = a.M * a.K / 16;
      int64_t blocks = (n16 + 255) / 256;
      if (blocks > 4096) blocks = 4096;
      cudaError_t e = launch_pdl(act_i8_to_f16_kernel, dim3(static_cast<unsigned>(blocks)),
                                 dim3(256), 0, stream, static_cast<const int8_t*>(a.act), dst, n16);
      if (e != cudaSuccess) return e;
      act16 = dst;
    }
  }
  CUtensorMap tw, ta;
  const uint64_t words_rows = static_cast<uint64_t>(a.K) / (C::kInt4 ? 8 : 4);
  if (a.wtiles != nullptr) {
    std::memset(&tw, 0, sizeof(tw));   // not read: the tiles come by bulk copies
  } else if (!make_map_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_INT32, a.qweight, a.N, words_rows,
                          static_cast<uint64_t>(a.N) * 4, kTileF, C::kWordRows,
                          CU_TENSOR_MAP_SWIZZLE_NONE)) {
    return cudaErrorInvalidValue;
  }
  if constexpr (!C::kXConv) {
    if (!make_act_map(&ta, C::kWO ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                      act16, a.M, a.K, T, 2 * GPS))
      return cudaErrorInvalidValue;
  } else {
    // int8 q_a [M][K]: one box is a 128-wide group of T rows, 128-byte swizzled
    if (!make_map_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, act8, a.K, a.M, a.K, kGroup, T,
                     CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  CUtensorMap ts;
  // scale rows per 128-wide group and per chunk load: W8A16 group-32 has 4,
  // group-128 one, per-column scales one row for all K
  const int s_rps = kMode != kModeW8A16 ? 1 : (a.group_size == 32 ? 4 : a.group_size == 128 ? 1 : 0);
  const uint32_t s_box = kMode != kModeW8A16 ? static_cast<uint32_t>(kScaleChunk * GPS)
                         : (s_rps == 0 ? 1u : static_cast<uint32_t>(kScaleChunk * s_rps));
  const uint64_t s_rows = kMode != kModeW8A16 ? static_cast<uint64_t>(a.K / kGroup)
                          : (a.group_size == 0 ? 1u : static_cast<uint64_t>(a.K / a.group_size));
  if constexpr (C::kScales) {
    if (!make_map_2d(&ts, C::kWO ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                     a.scales, a.N, s_rows, static_cast<uint64_t>(a.N) * 2, kTileF, s_box,
                     CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
  } else {
    ts = tw;  // not read
  }

  const uint32_t fixed = 1024 + C::kXSlots * C::kABytes + C::kXiSlots * C::kXiBytes +
                         C::kScaleBytes + kCtrlBytes + kArgBytes;
  int stages = static_cast<int>((kSmemLimit - fixed) / C::kStageBytes);
  if (stages > kMaxStages) stages = kMaxStages;
  const uint32_t smem = fixed + static_cast<uint32_t>(stages) * C::kStageBytes;

  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(qlin_gemm_kernel<kMode, T, GPS>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(kSmemLimit));
  });
  if (attr_err != cudaSuccess) return attr_err;

  KParams kp;
  kp.amax_keys = a.amax_keys;
  kp.wtiles = reinterpret_cast<const uint8_t*>(a.wtiles);
  kp.groups = a.K / kGroup;
  kp.s_rps = s_rps;
  kp.s_tx = s_box * 256u;
  kp.s_a = a.s_a;
  kp.out = a.out;
  kp.M = a.M;
  kp.N = a.N;
  kp.G = pl.G;
  kp.F = pl.F;
  kp.W = pl.steps;
  kp.TT = pl.TT;
  kp.band = pl.band;
  kp.counters = static_cast<int*>(a.workspace);
  kp.part = reinterpret_cast<float*>(static_cast<uint8_t*>(a.workspace) + pl.counter_bytes);
  kp.err = err;
  kp.limit_ns = kWaitLimitNs;
  kp.stages = stages;
  return launch_pdl(qlin_gemm_kernel<kMode, T, GPS>, dim3(static_cast<unsigned>(pl.ctas)),
                    dim3(C::kThreads), smem, stream, tw, ta, ts, kp);
}

template <int kMode>
cudaError_t launch_mode(const GemmArgs& a, const GemmPlan& pl, int* err, cudaStream_t stream) {
  switch (pl.T) {
    case 16:
      if (kMode == kModeW4 && a.K % 256 == 0) return launch_t<kMode, 16, kMode == kModeW4 ? 2 : 1>(a, pl, err, stream);
      return launch_t<kMode, 16, 1>(a, pl, err, stream);
    case 32:
      if (kMode == kModeW4 && a.K % 256 == 0) return launch_t<kMode, 32, kMode == kModeW4 ? 2 : 1>(a, pl, err, stream);
      return launch_t<kMode, 32, 1>(a, pl, err, stream);
    case 64:
      if (kMode == kModeW4 && a.K % 256 == 0 && pl.TT * pl.F * (pl.G / 2) >= 16 * pl.ctas)
        return launch_t<kMode, 64, kMode == kModeW4 ? 2 : 1>(a, pl, err, stream);
      return launch_t<kMode, 64, 1>(a, pl, err, stream);
    default: return launch_t<kMode, 96, 1>(a, pl, err, stream);
  }
}

}  // namespace

cudaError_t launch_argmax_finalize(const unsigned long long* keys, int64_t M, int32_t* idx,
                                   cudaStream_t stream) {
  const unsigned blocks = static_cast<unsigned>((M + 127) / 128);
  return launch_pdl(argmax_finalize_kernel, dim3(blocks), dim3(128), 0, stream, keys, M, idx);
}

GemmPlan plan_gemm(int64_t M, int64_t N, int64_t K, int sm_count) {
  GemmPlan p{};
  // Batches above 64 rows take 96-token tiles.  128-token tiles are not
  // planned: at M = 2048 and 8192 they ran the W8A8 MLP projections 3-12%
  // slower (two D buffers per group instead of four), and graph replays of
  // the 128-token-tile path ended in an unexplained launch failure.
  p.T = M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : 96;
  p.F = (N + kTileF - 1) / kTileF;
  p.TT = (M + p.T - 1) / p.T;
  p.G = K / kGroup;
  p.steps = p.TT * p.F * p.G;
  // At least kMinSteps (tile, group) steps per block: small layers use fewer
  // blocks instead of splitting every tile across many of them.
  const int64_t by_work = (p.steps + kMinSteps - 1) / kMinSteps;
  p.ctas = by_work < sm_count ? by_work : sm_count;
  if (p.ctas > static_cast<int64_t>(kArgmaxKeysOffset / sizeof(int)))
    p.ctas = static_cast<int64_t>(kArgmaxKeysOffset / sizeof(int));
  if (p.ctas < 1) p.ctas = 1;
  // Batches of many token tiles take whole tiles in bands instead (StepIter):
  // a band's 16-bit activations, about kBandBytes, stay in L2 while every
  // feature tile passes over them, and the blocks running together share
  // each weight tile.  No tile is split, so there is no fix-up.
  p.band = 0;
  if (p.TT >= kBandMinTiles) {
    const int64_t tile_bytes = static_cast<int64_t>(p.T) * K * 2;
    int64_t band = kBandBytes / tile_bytes;
    if (band < 1) band = 1;
    if (band > p.TT) band = p.TT;
    p.band = band;
    const int64_t tiles = p.TT * p.F;
    p.ctas = tiles < sm_count ? tiles : sm_count;
  }
  // One arrival counter per block: a tile split across blocks is counted on
  // the counter of its first contributing block, and a block is the first
  // contributor of at most one split tile (the tile its range ends in).  The
  // counters sit in a fixed region at the start of the workspace, so calls of
  // any shape that share a workspace never see each other's partials there.
  p.counter_bytes = kCounterBytes;
  const size_t partial_bytes = static_cast<size_t>(p.ctas) * 2 * p.T * kTileF * sizeof(float);
  // then the W8A8 activations in the code width the kernel reads, when the
  // caller's is the other one (1 KB aligned): the fp16 image of int8 codes
  // for token tiles of 64 and more, the int8 codes of fp16 ones below
  p.act_offset = (p.counter_bytes + partial_bytes + 1023) & ~static_cast<size_t>(1023);
  p.workspace_bytes = p.act_offset +
                      static_cast<size_t>(M) * static_cast<size_t>(K) * (p.T >= 64 ? 2 : 1);
  return p;
}

cudaError_t launch_gemm(const GemmArgs& a, const GemmPlan& p, int* err, cudaStream_t stream) {
  switch (a.mode) {
    case GemmMode::kW8A8: return launch_mode<kModeW8A8>(a, p, err, stream);
    case GemmMode::kW8A8Partials: return launch_mode<kModeP>(a, p, err, stream);
    case GemmMode::kW8A16: return launch_mode<kModeW8A16>(a, p, err, stream);
    default: return launch_mode<kModeW4>(a, p, err, stream);
  }
}

}  // namespace qlin
