/*
 * qlin.h -- C ABI of libqlin, group-wise quantized linear layers for GB300.
 *
 * The library implements the quantized linear layer used to serve quantized
 * block-diffusion drafters and their targets:
 *
 *   1. dynamic per-token symmetric INT8 activation quantization,
 *   2. a W8A8 GEMM against GPTQ-packed symmetric INT8 weights with one fp16
 *      scale per 128-wide K group (GS128),
 *   3. the W4A16 g128 symmetric weight-only GEMM with bf16 activations, and
 *      its int8 sibling W8A16 (group-32, group-128 or per-column scales),
 *   4. the GPTQ packer that produces the weight format of 2 and 3,
 *   5. the vocabulary head with fused greedy argmax (2 or 3 reduced to the
 *      largest output per row),
 *   6. the ingest of the compressed-tensors per-output-row packed orientation.
 *
 * Format (all calls): GPTQ qweight / qzeros / scales, no g_idx,
 * desc_act = false, symmetric, groups of exactly 128 contiguous K
 * ("Flint-DFlash2-GPTQ-INT8-PTQR" model card, parameter table and the text
 * under it; "Qwen3.8-27B-DFlash2-W4A16-g128-sym-GPTQ" card, property table).
 * There is no zero-point input and no bias: qzeros is produced by the packer
 * for format fidelity only and is never read.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Pointers are DEVICE pointers owned by the caller; the library never
 *    allocates, frees or retains them.  All matrices are dense row-major.
 *  - bf16 and fp16 values are passed as their 16-bit patterns (uint16_t).
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream) and returns a qlin_status_t at launch time.  Errors found
 *    on the device (a bounded wait that ran out, a packer input out of range)
 *    are recorded in a device-wide error word and reported by
 *    qlin_device_status().
 *  - No exception crosses the ABI and nothing is printed.
 *  - Shapes: M = tokens (rows of the activation), K = input features,
 *    N = output features.  K must be a positive multiple of 128, N a positive
 *    multiple of 8, M >= 0, and M, N, K <= 2^31 - 1.  M == 0 (an empty
 *    batch) reads and writes nothing and returns QLIN_OK after the shape
 *    checks; the pointers sized by M (activations, their scales, outputs)
 *    may then be NULL.
 *  - Alignment: every pointer must be 16-byte aligned (the kernels move data
 *    with TMA and 16-byte vector accesses), unless a call states otherwise.
 *  - The calls run only on an sm_103 GPU (GB300); elsewhere they return
 *    QLIN_ERR_DEVICE.
 */
#ifndef QLIN_H
#define QLIN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int qlin_status_t;

#define QLIN_OK                   0
#define QLIN_ERR_NULL            -1   /* a required pointer is NULL */
#define QLIN_ERR_SHAPE           -2   /* M, N or K outside the rules above */
#define QLIN_ERR_ALIGN           -3   /* a pointer is not 16-byte aligned */
#define QLIN_ERR_WORKSPACE       -4   /* workspace NULL or smaller than qlin_workspace_bytes() */
#define QLIN_ERR_BITS            -5   /* bits is not 4 or 8 */
#define QLIN_ERR_DEVICE          -6   /* the current device is not an sm_103 GPU */
#define QLIN_ERR_TOO_LARGE       -7   /* the problem needs more scratch than the no-alloc entry holds */
#define QLIN_ERR_CUDA           -10   /* a CUDA runtime call or kernel launch failed */
#define QLIN_ERR_DEVICE_TIMEOUT -20   /* a bounded wait inside a kernel ran out (device error word) */
#define QLIN_ERR_VALUE_RANGE    -21   /* the packer met a value outside the bit width (device error word) */

/* A cudaStream_t, declared without the CUDA headers. */
typedef struct CUstream_st *qlin_stream_t;

/*
 * Dynamic per-token symmetric INT8 activation quantization.
 *
 * Passages: "Flint-DFlash2-GPTQ-INT8-PTQR" card, PTQR paragraph ("dynamic
 * per-token activation quantization") and the serving recipe
 * (VLLM_GFX908_ACT_QUANT=round); "Qwen3.8-27B-GPTQ-INT8-W8A8-GS128-PTQR"
 * card, "Serving" (GEMM inputs are dynamically quantized to INT8).
 *
 * For each row m of x:  amax = max_k |x[m,k]|,  s_a[m] = amax / 127 (fp32,
 * IEEE divide),  q[m,k] = rint(x[m,k] / s_a[m]) (fp32 IEEE divide, ties to
 * even), clamped to [-127, 127].  A row of zeros gives s_a = 0 and q = 0.
 * Non-finite inputs are outside the contract.
 *
 *   x    bf16 [M, K]   input activations
 *   q    int8 [M, K]   output, quantized activations
 *   s_a  fp32 [M]      output, per-token scales
 */
qlin_status_t qlin_act_quant_i8(const uint16_t *x, int64_t M, int64_t K,
                                int8_t *q, float *s_a, qlin_stream_t stream);

/*
 * The producers of the projections' inputs, fused with the act-quant above:
 * one read of the producer's input and one write of q and s_a.
 *
 * Passages: "Qwen3.8-27B-DFlash2-W4A16-g128-sym-GPTQ" card, the table of
 * components kept in BF16 (input_layernorm, post_attention_layernorm: the
 * RMSNorms in front of the q/k/v and gate/up projections) and the linear-layer
 * table (mlp.{gate,up,down}_proj: down_proj reads SiLU(gate) * up); the
 * act-quant passages above.
 *
 * qlin_rmsnorm_act_quant_i8, for each row m of x:
 *   variance = mean_k x[m,k]^2 (fp32),  rstd = 1 / sqrt(variance + eps)
 *   (IEEE square root and divide),  t = bf16(x * rstd),
 *   z[m,k] = bf16(gamma[k] * t)  (the decoder norm's bf16 output),
 * then (q, s_a) = act-quant of z exactly as qlin_act_quant_i8 defines it.
 *   x      bf16 [M, K]   the residual stream
 *   gamma  bf16 [K]      the norm's weight
 *   eps    >= 0, finite
 *
 * qlin_silu_mul_act_quant_i8, for each row m of gate_up [M, 2I] (the fused
 * gate/up projection's output: gate in columns [0, I), up in [I, 2I)):
 *   z[m,i] = bf16(SiLU(g) * u),  SiLU(g) = g * sigmoid(g) in fp32, the
 *   sigmoid from e = expf(-|g|) and an approximate divide by 1 + e (within
 *   2 ulp), g = gate_up[m,i], u = gate_up[m,I+i],
 * then (q, s_a) = act-quant of z.
 *
 *   q    int8 [M, K] (or [M, I])   output
 *   s_a  fp32 [M]                  output
 *   y    bf16 [M, K] (or [M, I])   optional output: z itself; NULL skips it
 *
 * K (or I) must be a positive multiple of 128; all pointers 16-byte aligned.
 * Non-finite inputs are outside the contract.
 */
qlin_status_t qlin_rmsnorm_act_quant_i8(const uint16_t *x, const uint16_t *gamma, float eps,
                                        int64_t M, int64_t K, int8_t *q, float *s_a,
                                        uint16_t *y, qlin_stream_t stream);

qlin_status_t qlin_silu_mul_act_quant_i8(const uint16_t *gate_up, int64_t M, int64_t I,
                                         int8_t *q, float *s_a, uint16_t *y,
                                         qlin_stream_t stream);

/*
 * The three producers above with the codes written as fp16 instead of int8:
 * q[m,k] is the same integer in [-127, 127], stored as its (exact) fp16 value,
 * fp16 [M, K] (or [M, I]).  s_a and y as above.
 *
 * The passages are those of the producers above; the width of the codes is
 * a storage choice of this library.  qlin_gemm_w8a8_gs128_c16 reads these
 * codes: for batches of more than 32 tokens its tensor-core operands are the
 * fp16 codes themselves, so handing them over directly saves the conversion
 * pass that the int8 entry runs first.  The results are bit-identical to the
 * int8 pair (qlin_*_i8 followed by qlin_gemm_w8a8_gs128).
 */
qlin_status_t qlin_act_quant_c16(const uint16_t *x, int64_t M, int64_t K,
                                 uint16_t *q, float *s_a, qlin_stream_t stream);

qlin_status_t qlin_rmsnorm_act_quant_c16(const uint16_t *x, const uint16_t *gamma, float eps,
                                         int64_t M, int64_t K, uint16_t *q, float *s_a,
                                         uint16_t *y, qlin_stream_t stream);

qlin_status_t qlin_silu_mul_act_quant_c16(const uint16_t *gate_up, int64_t M, int64_t I,
                                          uint16_t *q, float *s_a, uint16_t *y,
                                          qlin_stream_t stream);

/*
 * W8A8 GS128 linear:  y = bf16( s_a[m] * sum_g s_w[g,n] * P[g,m,n] ),
 * P[g,m,n] = sum_{k = 128g}^{128g+127} q_a[m,k] * q_w[k,n]  (exact integers).
 *
 * Passages: "Qwen3.8-27B-GPTQ-INT8-W8A8-GS128-PTQR" card, "Quantization
 * details" (true int8 x int8 compute at every decode and prefill GEMM shape,
 * one weight scale per 128-wide K block); "Flint-DFlash2-GPTQ-INT8-PTQR"
 * card, parameter table and the "AITER W8A8 INT8 GEMMs at every M" contract.
 *
 * Each group's partial P is computed exactly; groups are rescaled in fp32 by
 * fma(P, s_w, acc) in ascending g, the result is multiplied once by s_a[m]
 * and rounded to bf16 (nearest even).  When K is split across thread blocks
 * the per-split fp32 partials are summed in ascending split order, so the
 * result is deterministic for a given (M, N, K) and device.
 *
 *   q_a      int8  [M, K]          quantized activations (qlin_act_quant_i8)
 *   s_a      fp32  [M]             activation scales
 *   qweight  int32 [K/4, N]        GPTQ words: byte i of word (kk, n) holds
 *                                  q_w[4kk+i, n] + 128, byte 0 least significant
 *   scales   fp16  [K/128, N]      weight group scales s_w
 *   y        bf16  [M, N]          output
 *   workspace / workspace_bytes    at least qlin_workspace_bytes(M, N, K) bytes
 *            of device memory, ZEROED BEFORE ITS FIRST USE.  It holds split-K
 *            partials and arrival counters; the kernels return the counters to
 *            zero, so the buffer can be reused by later calls that are ordered
 *            on one stream.  Calls that share a workspace must not overlap.
 *            After a device error (QLIN_ERR_DEVICE_TIMEOUT) zero it again.
 */
qlin_status_t qlin_gemm_w8a8_gs128(const int8_t *q_a, const float *s_a,
                                   const int32_t *qweight, const uint16_t *scales,
                                   int64_t M, int64_t N, int64_t K, uint16_t *y,
                                   void *workspace, size_t workspace_bytes,
                                   qlin_stream_t stream);

/*
 * qlin_gemm_w8a8_gs128 with the activation codes as fp16 (the output of the
 * qlin_*_c16 producers): q_a fp16 [M, K], every value an integer in
 * [-127, 127]; other values are outside the contract.  Same results, same
 * workspace size.  Batches of up to 32 tokens, whose kernel reads int8
 * codes, first narrow the codes into the workspace.
 */
qlin_status_t qlin_gemm_w8a8_gs128_c16(const uint16_t *q_a, const float *s_a,
                                       const int32_t *qweight, const uint16_t *scales,
                                       int64_t M, int64_t N, int64_t K, uint16_t *y,
                                       void *workspace, size_t workspace_bytes,
                                       qlin_stream_t stream);

/*
 * W8A8 GS128 linear for callers that cannot allocate device memory.
 *
 * The pages have no counterpart to this call; it exists for the library's
 * users.  Some callers cannot call cudaMalloc or hand the library a workspace
 * -- code running inside an allocator or memory-pool callback, a plugin whose
 * host framework owns every device allocation, or a process that must not
 * grow its device footprint once it is serving.  This call computes exactly
 * what qlin_gemm_w8a8_gs128 computes (same kernel, same split of K, same
 * results) but takes its scratch from a fixed 24 MiB array compiled
 * into the library, which every GPU that loads the library holds until the
 * process exits.  It allocates nothing.
 *
 *  - The first call on a device looks up the array's device address (with that
 *    device current) and caches it; make that first call before any stream
 *    capture.
 *  - Problems whose scratch need (qlin_workspace_bytes) exceeds 24 MiB return
 *    QLIN_ERR_TOO_LARGE; on a 152-SM GB300 every shape with M <= 96 and
 *    K <= 50,000 fits.
 *  - All calls share the one array, which keeps the last call's contents; the
 *    call clears the arrival counters with cudaMemsetAsync on `stream` before
 *    its kernel.  Calls that overlap on the GPU (other streams, unordered host
 *    threads) race on the array: order them on one stream.
 *
 * Arguments as for qlin_gemm_w8a8_gs128, without the workspace.
 */
qlin_status_t qlin_gemm_w8a8_gs128_noalloc(const int8_t *q_a, const float *s_a,
                                           const int32_t *qweight, const uint16_t *scales,
                                           int64_t M, int64_t N, int64_t K, uint16_t *y,
                                           qlin_stream_t stream);

/*
 * W4A16 g128 symmetric weight-only linear:
 *   w[k,n] = bf16( q_w[k,n] * s[k/128, n] ),   y = bf16( sum_k x[m,k] * w[k,n] )
 * accumulated in fp32.
 *
 * Passages: "Qwen3.8-27B-DFlash2-W4A16-g128-sym-GPTQ" card, property table
 * (4-bit weights, BF16 activations, group_size=128, symmetric; INT32-packed)
 * and the apply_dense_kv_fix format table (W4A16 GPTQ: unpack_from_int32 +
 * group scales).
 *
 *   x        bf16  [M, K]          activations
 *   qweight  int32 [K/8, N]        nibble i (bits 4i..4i+3) of word (kk, n)
 *                                  holds q_w[8kk+i, n] + 8
 *   scales   bf16  [K/128, N]      group scales
 *   y        bf16  [M, N]          output
 *   workspace / workspace_bytes    as for qlin_gemm_w8a8_gs128
 */
qlin_status_t qlin_gemm_w4a16_g128(const uint16_t *x, const int32_t *qweight,
                                   const uint16_t *scales, int64_t M, int64_t N,
                                   int64_t K, uint16_t *y, void *workspace,
                                   size_t workspace_bytes, qlin_stream_t stream);

/*
 * The weights in the tile layout: the same GPTQ words, reordered once (at
 * load time) so that the GEMM's weight stream reads each step's tile as one
 * contiguous block.  Tile (f, g) holds the words of output features
 * 128f..128f+127 and K group g (K values 128g..128g+127): W x 128 int32, W =
 * 32 words for 8-bit and 16 for 4-bit weights, word (kk, j) of the tile =
 * qweight[g*W + kk][128f + j]; tiles follow each other by f, then g.  Words
 * of features at or past N (the last tile, when N is not a multiple of 128)
 * are 0 and never reach an output.
 *
 * Passages: "Qwen3.8-27B-DFlash2-W4A16-g128-sym-GPTQ" card, property table
 * ("compressed-tensors pack-quantized (Marlin-compatible)": serving kernels
 * take GPTQ words reordered for their own access pattern); the GPTQ format
 * of the "Flint-DFlash2-GPTQ-INT8-PTQR" card.  The reordering is this
 * library's own.
 *
 * qlin_tiles_bytes: bytes of the tile layout, ceil(N/128) * 128 * K * bits /
 *   8; 0 for an invalid shape or bits.
 * qlin_pack_tiles:
 *   qweight  int32 [K*bits/32, N]  GPTQ words (device, 16-byte aligned)
 *   bits     8 or 4
 *   tiles    int32, qlin_tiles_bytes(K, N, bits) bytes (device, 16-byte
 *            aligned, caller-owned)
 *   Asynchronous on `stream`.  Errors: QLIN_ERR_NULL, QLIN_ERR_BITS,
 *   QLIN_ERR_SHAPE (K a positive multiple of 128, N >= 1), QLIN_ERR_ALIGN.
 *
 * qlin_gemm_w8a8_gs128_tiled / qlin_gemm_w4a16_g128_tiled: the same linears
 * as qlin_gemm_w8a8_gs128 / qlin_gemm_w4a16_g128, bit for bit, with the
 * weights in the tile layout (`tiles`, from qlin_pack_tiles with bits 8 / 4)
 * in place of qweight.  All other arguments, errors and the workspace are as
 * for those calls.
 */
size_t qlin_tiles_bytes(int64_t K, int64_t N, int bits);
qlin_status_t qlin_pack_tiles(const int32_t *qweight, int64_t K, int64_t N, int bits,
                              int32_t *tiles, qlin_stream_t stream);
qlin_status_t qlin_gemm_w8a8_gs128_tiled(const int8_t *q_a, const float *s_a,
                                         const int32_t *tiles, const uint16_t *scales,
                                         int64_t M, int64_t N, int64_t K, uint16_t *y,
                                         void *workspace, size_t workspace_bytes,
                                         qlin_stream_t stream);
qlin_status_t qlin_gemm_w4a16_g128_tiled(const uint16_t *x, const int32_t *tiles,
                                         const uint16_t *scales, int64_t M, int64_t N,
                                         int64_t K, uint16_t *y, void *workspace,
                                         size_t workspace_bytes, qlin_stream_t stream);

/*
 * W8A16 int8 weight-only linear, bf16 activations:
 *   w[k,n] = bf16( q_w[k,n] * s[k / group_size, n] ),   y = bf16( sum_k x[m,k] * w[k,n] )
 * accumulated in fp32 (one rounding of each exact product q * s).
 *
 * Passages: "Qwen3.5-4B-DFlash-W8A16" card (a weight-only int8 drafter, RTN
 * on the weights, bf16 activations); "DFlash2 decoding" recipe page (int8
 * drafter projections with group-32 scales).
 *
 *   x           bf16  [M, K]             activations
 *   qweight     int32 [K/4, N]           8-bit GPTQ words as for the W8A8 GEMM
 *                                        (byte i of word (kk, n) = q_w[4kk+i, n] + 128)
 *   scales      bf16  [K/group_size, N]  group scales, or [1, N] for group_size 0
 *   group_size  32, 128, or 0 (one scale per output column)
 *   y           bf16  [M, N]             output
 *   workspace / workspace_bytes          as for qlin_gemm_w8a8_gs128
 *
 * Any other group_size returns QLIN_ERR_SHAPE.
 */
qlin_status_t qlin_gemm_w8a16(const uint16_t *x, const int32_t *qweight, const uint16_t *scales,
                              int64_t M, int64_t N, int64_t K, int group_size, uint16_t *y,
                              void *workspace, size_t workspace_bytes, qlin_stream_t stream);

/*
 * Vocabulary head with fused greedy argmax: the same linear as
 * qlin_gemm_w8a8_gs128 / qlin_gemm_w4a16_g128, but instead of y the call
 * returns, per row m, the column index of the largest bf16 output value (the
 * lowest index on ties; -0 equals +0).  y itself is never written.
 *
 * Passages: "DFlash2 decoding" recipe page (Eole), which runs single-GPU,
 * batch-one greedy inference with an INT8 or INT4 group-128 shared
 * vocabulary head; the Flint card's INT8 LM head switch.  Greedy decoding
 * needs only the argmax.
 *
 *   arguments as for the matching GEMM, except:
 *   argmax   int32 [M]             device; 4-byte aligned
 *   M        at most 96 (one token tile); larger M returns QLIN_ERR_SHAPE
 *   workspace / workspace_bytes    at least qlin_workspace_bytes(M, N, K)
 *
 * Each output value is the bit-identical bf16 value the matching GEMM call
 * writes for the same (M, N, K) on the same device, so the index equals the
 * argmax of that call's y.  Asynchronous on `stream`.  Calls that share a
 * workspace must not overlap.
 */
qlin_status_t qlin_gemm_w8a8_gs128_argmax(const int8_t *q_a, const float *s_a,
                                          const int32_t *qweight, const uint16_t *scales,
                                          int64_t M, int64_t N, int64_t K, int32_t *argmax,
                                          void *workspace, size_t workspace_bytes,
                                          qlin_stream_t stream);
qlin_status_t qlin_gemm_w4a16_g128_argmax(const uint16_t *x, const int32_t *qweight,
                                          const uint16_t *scales, int64_t M, int64_t N,
                                          int64_t K, int32_t *argmax, void *workspace,
                                          size_t workspace_bytes, qlin_stream_t stream);

/*
 * GPTQ packer (offline step; not on the timed path).
 *
 * Passages: "Flint-DFlash2-GPTQ-INT8-PTQR" card, parameter table (GPTQ
 * qweight/qzeros/scales, INT8, symmetric, no g_idx);
 * "Qwen3.8-27B-DFlash2-W4A16-g128-sym-GPTQ" card (INT32-packed 4-bit weights).
 *
 *   q        int8  [K, N]          weights, in [-2^(bits-1), 2^(bits-1) - 1]
 *   bits     8 or 4
 *   qweight  int32 [K*bits/32, N]  output: field i of word (kk, n) holds
 *                                  q[(32/bits)*kk + i, n] + 2^(bits-1),
 *                                  field 0 least significant
 *   qzeros   int32 [K/128, N*bits/32] output or NULL; every field = 2^(bits-1)
 *                                  (needs N*bits % 32 == 0 when not NULL)
 * A value outside the range is packed masked and flags QLIN_ERR_VALUE_RANGE
 * in the device error word.
 */
qlin_status_t qlin_pack_gptq(const int8_t *q, int64_t K, int64_t N, int bits,
                             int32_t *qweight, int32_t *qzeros, qlin_stream_t stream);

/*
 * Ingest of the compressed-tensors "pack-quantized" orientation, the native
 * format of the "Qwen3.8-27B-DFlash2-W4A16-g128-sym-GPTQ" card (property
 * table, Format row).  There the packed weight is stored per output row:
 * word (n, kk) holds the same fields as GPTQ word (kk, n) (field i =
 * q_w[(32/bits) kk + i, n] + 2^(bits-1), field 0 least significant), and the
 * scales are [N, K/128].  This call transposes both, bit for bit, into the
 * orientation the GEMMs read (offline step; not on the timed path).
 *
 *   packed_nk  int32 [N, K*bits/32]   device, 4-byte aligned
 *   scales_ng  16-bit [N, K/128]      device, 2-byte aligned (bf16 or fp16 bits)
 *   bits       4 or 8
 *   qweight    int32 [K*bits/32, N]   output, device, 16-byte aligned
 *   scales     16-bit [K/128, N]      output, device, 16-byte aligned
 *
 * K must be a multiple of 128.  Asynchronous on `stream`.
 */
qlin_status_t qlin_ingest_nk(const int32_t *packed_nk, const uint16_t *scales_ng, int64_t K,
                             int64_t N, int bits, int32_t *qweight, uint16_t *scales,
                             qlin_stream_t stream);

/*
 * Bytes of workspace the GEMMs need for (M, N, K) on the current device: a
 * fixed region of arrival counters (one per block), the fp32 split-K
 * partials of two output tiles per block, and, for token tiles of 64 and
 * more (M > 32), the fp16 image of the W8A8 activations.  Returns 0 for
 * shapes the GEMMs reject.
 */
size_t qlin_workspace_bytes(int64_t M, int64_t N, int64_t K);

/*
 * Test hook: the exact per-group integer partials of the W8A8 path,
 * P[g, m, n] (int32 [K/128, M, N]), produced by the same tensor-core pipeline
 * as qlin_gemm_w8a8_gs128 (exactly-converted int8 operands, fp32 TMEM
 * accumulation of one 128-wide group), read back without rescaling.
 * Meant for small shapes.  workspace as for the GEMM.
 */
qlin_status_t qlin_debug_group_partials_i8(const int8_t *q_a, const int32_t *qweight,
                                           int64_t M, int64_t N, int64_t K,
                                           int32_t *P, void *workspace,
                                           size_t workspace_bytes, qlin_stream_t stream);

/*
 * Test hook: launches one block whose thread waits on a barrier that nothing
 * completes, with a wait limit of limit_ns nanoseconds (1e3 .. 1e10).  The
 * wait runs out, the kernel records QLIN_ERR_DEVICE_TIMEOUT in the device
 * error word and returns normally; the CUDA context stays usable.
 */
qlin_status_t qlin_debug_wait_timeout(int64_t limit_ns, qlin_stream_t stream);

/*
 * Synchronizes `stream`, then reads and clears the device-wide error word of
 * the current device.  Returns QLIN_OK, QLIN_ERR_DEVICE_TIMEOUT,
 * QLIN_ERR_VALUE_RANGE, or QLIN_ERR_CUDA if the synchronization failed.
 */
qlin_status_t qlin_device_status(qlin_stream_t stream);

/*
 * The device error word without clearing it: returns the status
 * qlin_device_status would return and, when it is not QLIN_OK, the code
 * location of the failing wait or check (`where`, a small integer naming the
 * role and the wait inside the kernel) and the index of the thread block that
 * recorded it.  Synchronizes `stream`.  Either output may be NULL.
 */
qlin_status_t qlin_device_error_detail(qlin_stream_t stream, int32_t *where, int32_t *block);

/* A static, human-readable name for a status code. */
const char *qlin_status_string(qlin_status_t status);

/* Library ABI version (major * 100 + minor).  1.1 (101) adds the W8A16
 * GEMM, the greedy-argmax GEMMs, the compressed-tensors ingest, the fused
 * producers and qlin_device_error_detail to the 1.0 calls; no 1.0 call
 * changed, except that an empty batch (M == 0) now accepts NULL batch
 * buffers.  1.2 (102) adds the tile layout (qlin_tiles_bytes,
 * qlin_pack_tiles) and the tiled W8A8 and W4A16 GEMMs; the greedy-argmax
 * calls now take at most 96 rows.  1.3 (103) adds the fp16 activation codes
 * (qlin_act_quant_c16, qlin_rmsnorm_act_quant_c16,
 * qlin_silu_mul_act_quant_c16, qlin_gemm_w8a8_gs128_c16); the workspace of
 * batches of up to 32 tokens grows by M * K bytes. */
int qlin_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QLIN_H */
