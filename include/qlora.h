/*
 * qlora.h -- C ABI of the B300 (sm_103a) QLoRA NF4 linear-layer library.
 *
 * The library implements the hot path of a QLoRA linear layer:
 *   - blockwise NF4 quantisation of a frozen base weight with double
 *     quantisation of the block constants,
 *   - dequantisation of that weight to bf16,
 *   - the forward pass  y = x . W_hat^T + (x . A^T) . B^T . alpha / r
 *     (a fused dequantise + tensor-core GEMM for M > 16 tokens, a
 *     memory-bound decode GEMV streaming the packed weights for M <= 16;
 *     both compute with the exact bf16 W_hat the dequantiser produces),
 *   - the backward pass dX, dA and dB with the NF4 buffers frozen.
 *
 * Sources of each operation (page title -- section):
 *   [QLoRA-26]  "QLoRA and 4bit Quantization | QLoRA 与 4-bit 量化" (datawhale ch. 26)
 *   [QLoRA-22]  "QLoRA and 4bit Quantization | QLoRA 与 4-bit NormalFloat 量化核心机制"
 *               (datawhale ch. 22)
 *   [Gemma-9]   "第 09 期 | QLoRA 4-bit 量化微调：消费级显卡也能训" (agentupdate gemma lesson 9)
 *   [Finetune-4] "QLoRA 的三个核心技术" (gufacode finetune ch. 4)
 *
 * Conventions shared by every entry point:
 *   - Every pointer named "device" is a device (HBM) address owned by the
 *     caller.  The library never allocates, frees or retains memory.
 *   - Row-major storage.  x, dY, y and dX are [M, features] with any leading
 *     batch dimensions flattened into M.
 *   - bf16 values travel as their 16-bit patterns (uint16_t).
 *   - Every compute call is asynchronous on `stream` (a cudaStream_t passed
 *     as void*; NULL is the legacy default stream).  The returned status
 *     covers host-side argument validation and launch errors only.  Errors
 *     detected on the device (a pipeline wait that ran out, non-finite
 *     weights) are written to device words and read after synchronising
 *     (qlora_device_status, the quantiser's nonfinite flag).
 *   - Stream order holds as usual.  The forward and backward kernels are
 *     launched with programmatic dependent launch: one may start while the
 *     work before it on the stream finishes, but it touches no global memory
 *     until that work has completed and its writes are visible.
 *   - Device pointers must be 16-byte aligned.
 *   - The NF4 buffers are const in the forward and backward calls: that is
 *     the frozen-base contract ([QLoRA-26] Step 4 "frozen base gradient
 *     contract"); nothing is ever written to them after quantisation.
 *   - No bias on either branch ([QLoRA-26] Step 3 formula); LoRA dropout on
 *     the bypass input through the *_dropout calls below.
 */
#ifndef QLORA_B300_H
#define QLORA_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  QLORA_OK = 0,
  QLORA_ERR_INVALID_ARG = 1, /* null pointer, negative size, bad enum */
  QLORA_ERR_SHAPE = 2,       /* shape outside the supported set */
  QLORA_ERR_ALIGN = 3,       /* pointer or stride not 16-byte aligned */
  QLORA_ERR_DTYPE = 4,       /* dtype not supported for this argument */
  QLORA_ERR_NONFINITE = 5,   /* reserved for device-side non-finite report */
  QLORA_ERR_TIMEOUT = 6,     /* a bounded device wait ran out (device word) */
  QLORA_ERR_CUDA = 7,        /* a CUDA runtime call or launch failed */
  QLORA_ERR_WORKSPACE = 8    /* workspace missing or too small */
} qlora_status;

typedef enum { QLORA_F32 = 0, QLORA_BF16 = 1 } qlora_dtype;

/* The 16-entry table the indices point into.
 *   QLORA_CODEBOOK_PRINTED: the NF4 table printed by create_nf4_lookup_table
 *     ([QLoRA-26] Step 4, [QLoRA-22] Step 4): -1, -0.696, ..., 0, ..., 0.723, 1
 *     (each the fp32 nearest to the printed decimal; index 7 is zero).
 *   QLORA_CODEBOOK_QUANTILE: the construction of [QLoRA-26] Step 2,
 *     q_i = Phi^-1((i - 0.5) / 16), i = 1..16, divided by q_16 so that it
 *     runs from -1 to 1 (the page does not say how the quantiles are
 *     normalised; this is the library's reading); symmetric, no zero.  Phi^-1
 *     is Wichura's AS 241 in binary64, the upper half mirrored. */
typedef enum { QLORA_CODEBOOK_PRINTED = 0, QLORA_CODEBOOK_QUANTILE = 1 } qlora_codebook;

/* A quantised weight W_hat of logical shape [rows, cols] = [N out, K in].
 *
 * [Gemma-9] 9.2.1 and [QLoRA-22] "engineering notes": the weight is cut into
 * blocks of `block` consecutive elements of the row-major flattened matrix
 * (cols % block == 0, so a block never crosses a row); each block is
 * normalised by its absolute maximum and every element is stored as the
 * 4-bit index of the nearest entry of the 16-entry NF4 table ([QLoRA-26]
 * Step 2 and Step 4 create_nf4_lookup_table).
 * [QLoRA-22] QLoRALinearSim docstring: two 4-bit indices share one byte.
 * Element 2j sits in the HIGH nibble of byte j, element 2j+1 in the LOW
 * nibble (the pages fix no order; this is the library's convention).
 * [Gemma-9] 9.2.2 and [Finetune-4] "double quantization": the block
 * absmax constants are quantised again to 8 bits.  `group` consecutive
 * block constants share one fp32 scale s2 = max/127; each constant is stored
 * as the int8 clamp(rint_even(absmax / s2), -127, 127).  group == 0 keeps
 * the constants in fp32 (absmax_f32) instead.
 *
 * Sizes (qlora_nf4_sizes): packed rows*cols/2 bytes; absmax_code nblocks
 * bytes (group > 0); absmax_f32 nblocks floats (group == 0); scale2
 * ceil(nblocks/group) floats (group > 0); nblocks = rows*cols/block.
 * Supported: block in {64, 128} ([QLoRA-22] engineering notes: 64 or 128
 * weights share one scale); group in {0, 32, 64, 128, 256}; codebook a
 * qlora_codebook value (0, the printed table, when the struct is zeroed).
 * All pointers are device pointers owned by the caller; unused ones are NULL. */
typedef struct {
  int64_t rows;
  int64_t cols;
  int32_t block;
  int32_t group;
  int32_t codebook;  /* qlora_codebook */
  int32_t reserved;  /* 0 */
  uint8_t *packed;
  int8_t *absmax_code;
  float *absmax_f32;
  float *scale2;
} qlora_nf4_weight;

/* Byte counts of the three NF4 buffers of a [rows, cols] weight.
 * [QLoRA-26] Step 4 (qlora_trainable_state_ledger: packed size is numel/2
 * bytes) and [Finetune-4] (4.5 bits per parameter with fp32 constants,
 * about 4.127 with 8-bit constants).  Host only; any output may be NULL.
 * Returns QLORA_ERR_SHAPE for rows/cols < 0, block <= 0 or odd, cols % block,
 * or group < 0. */
qlora_status qlora_nf4_sizes(int64_t rows, int64_t cols, int32_t block, int32_t group,
                             size_t *packed_bytes, size_t *code_bytes, size_t *scale_bytes);

/* Quantise W (device, [rows, cols], fp32 or bf16 per w_dtype) into `out`.
 * [Gemma-9] 9.2.1-9.2.2, [QLoRA-26] Step 2 (0.20 -> 0.161), [Finetune-4].
 * Per block: a = max |w| over finite elements; each element's normalised
 * value w / a (IEEE fp32 division) is replaced by the index of the nearest
 * NF4 codepoint (fp32 distances, the lower index on an exact tie); a block
 * with a == 0 stores index 7 everywhere (the exact-zero codepoint of the
 * printed table; with the quantile table any index dequantises to 0 there).
 * The table is out->codebook.  Then the
 * double quantisation above.  `out` (host struct) describes caller-allocated
 * device buffers of the sizes from qlora_nf4_sizes.
 * nonfinite_flag: NULL, or a device int32 that the kernel sets to 1 when it
 * meets a NaN or infinite weight (the caller zeroes it first); indices of
 * such blocks are unspecified.  It is set to QLORA_ERR_TIMEOUT instead when
 * a copy of the weight into shared memory did not complete within the
 * kernel's time limit (about 2 s); all outputs are then unspecified.
 * Errors: QLORA_ERR_INVALID_ARG (null buffers), QLORA_ERR_SHAPE (block not 64
 * or 128, unsupported group, cols % block), QLORA_ERR_DTYPE, QLORA_ERR_ALIGN,
 * QLORA_ERR_CUDA. */
qlora_status qlora_quantize_nf4(const void *W, qlora_dtype w_dtype, const qlora_nf4_weight *out,
                                int32_t *nonfinite_flag, void *stream);

/* Dequantise `w` into W_out (device, bf16 patterns, [rows, cols]).
 * [QLoRA-26] Step 3/4 (table[index] * scale), [Gemma-9] 9.2.2 (the 8-bit
 * constants are dequantised first) and 9.3 (bf16 compute dtype):
 *   a_hat = float(code) * s2          (fp32 product; group > 0)
 *   a_hat = absmax_f32[block]         (group == 0)
 *   w_hat = bf16_round_nearest_even(codepoint[index] * a_hat)  (fp32 product)
 * Errors as for qlora_quantize_nf4. */
qlora_status qlora_dequant(const qlora_nf4_weight *w, uint16_t *W_out, void *stream);

/* Adapter merge: W_out = bf16(W_hat + (alpha / r) . B . A), [N, K] bf16.
 * [QLoRA-26] Step 5 conclusion (adapter merge and deployment loading are
 * what a trained adapter still has to pass) and [Select-65] (the merged
 * model as the delivered artifact).  The Step 3 forward formula gives
 *   x . W_hat^T + (x . A^T) . B^T . alpha / r = x . (W_hat + alpha/r . B . A)^T,
 * so the merged weight serves the same forward without the LoRA branch (up
 * to its one bf16 rounding).  Arithmetic: W_hat exactly as qlora_dequant
 * produces it, B . A with bf16 operands and fp32 accumulation, one fp32
 * multiply-add with alpha / r (fp32), one rounding to bf16.
 *   w      quantised base weight [N, K] (const)
 *   A      device bf16 [r, K];  B  device bf16 [N, r];  8 <= r <= 64, r % 8 == 0
 *   W_out  device bf16 [N, K], caller-owned
 * Errors: QLORA_ERR_INVALID_ARG, QLORA_ERR_SHAPE, QLORA_ERR_ALIGN, QLORA_ERR_CUDA. */
qlora_status qlora_merge_lora(const qlora_nf4_weight *w, const uint16_t *A, const uint16_t *B,
                              int32_t r, float alpha, uint16_t *W_out, void *stream);

/* Workspace bytes for qlora_linear_fwd / qlora_linear_bwd at these sizes
 * (M tokens, N out features, K in features, LoRA rank r) on the current
 * device.  One workspace sized this way serves both calls.  It includes a
 * split-tile area (fp32 partial tiles, 512 KiB per pair of SMs: 37 MiB on a
 * 148-SM device) that lets the fused GEMM spread a layer whose output tiles
 * do not fill the SMs' waves over all of them.  Host only. */
qlora_status qlora_workspace_size(int64_t M, int64_t N, int64_t K, int32_t r, size_t *bytes);

/* The least workspace the calls accept: qlora_workspace_size without the
 * split-tile area.  With less than qlora_workspace_size bytes the fused GEMM
 * computes whole output tiles only (same results, fewer busy SMs on some
 * shapes).  Host only. */
qlora_status qlora_workspace_size_min(int64_t M, int64_t N, int64_t K, int32_t r, size_t *bytes);

/* Zero a freshly allocated workspace (device).  Must be called once before
 * the first forward/backward call that uses it; the library keeps the parts
 * that must start at zero at zero after every call that completes.  After a
 * call whose device status is QLORA_ERR_TIMEOUT, zero it again. */
qlora_status qlora_workspace_init(void *ws, size_t ws_bytes, void *stream);

/* Read (and clear) the device status word of a workspace: synchronises
 * `stream`, copies the word to *status (QLORA_OK or QLORA_ERR_TIMEOUT). */
qlora_status qlora_device_status(void *ws, int32_t *status, void *stream);

/* Flags of qlora_linear_fwd: select the kernel explicitly (tests only).
 * Default (0): GEMV for M <= 16, tensor-core GEMM otherwise.  FORCE_GEMV
 * returns QLORA_ERR_SHAPE for M > 16 (or a K whose x slice does not fit the
 * decode kernel's shared memory). */
#define QLORA_FLAG_FORCE_GEMV 1u
#define QLORA_FLAG_FORCE_GEMM 2u

/* Forward of the QLoRA linear layer ([QLoRA-26] Step 3 formula, read as
 *   y = x . W_hat^T + (x . A^T) . B^T . alpha / r,
 * and Step 4 TODO 2: the base branch is a linear map by the dequantised
 * weight, the LoRA branch goes through A then B then the scaling).
 *   w      quantised base weight, [N, K]
 *   x      device bf16 [M, K]
 *   A      device bf16 [r, K]  (lora_A)
 *   B      device bf16 [N, r]  (lora_B)
 *   r      1 <= r <= 64 and r % 8 == 0;  alpha: scaling is alpha / r in fp32
 *   y      device [M, N], fp32 or bf16 per y_dtype
 *   t_save device fp32 [M, r] or NULL: receives t = x . A^T (fp32
 *          accumulation) for the backward pass
 *   ws     device workspace of qlora_workspace_size(M, N, K, r) bytes,
 *          zeroed once by qlora_workspace_init; it also holds the device
 *          status word
 * Requires K % block == 0, N % 8 == 0, M >= 1.  Arithmetic: bf16 operands,
 * fp32 accumulation.  Errors: QLORA_ERR_INVALID_ARG, QLORA_ERR_SHAPE,
 * QLORA_ERR_ALIGN, QLORA_ERR_DTYPE, QLORA_ERR_WORKSPACE, QLORA_ERR_CUDA. */
qlora_status qlora_linear_fwd(const qlora_nf4_weight *w, const uint16_t *x, int64_t M,
                              const uint16_t *A, const uint16_t *B, int32_t r, float alpha,
                              void *y, qlora_dtype y_dtype, float *t_save, void *ws,
                              size_t ws_bytes, uint32_t flags, void *stream);

/* Backward of the QLoRA linear layer.  [QLoRA-26] Step 3 and Step 4 test
 * "frozen base gradient contract": gradients reach x, A and B, never the NF4
 * state; [QLoRA-22] Step 1: the gradient flows through the dequantised base
 * weight to x.  With s = alpha / r and t = x . A^T:
 *   u  = dY . B                    [M, r]   (fp32, kept in the workspace)
 *   dX = dY . W_hat + s . u . A    [M, K]   (fp32 or bf16 per dx_dtype)
 *   dA = s . u^T . x               [r, K]   (fp32)
 *   dB = s . dY^T . t              [N, r]   (fp32)
 *   dY      device bf16 [M, N];  x, A, B as in the forward
 *   t_saved device fp32 [M, r] from the forward, or NULL (recomputed)
 *   dX, dA, dB device outputs (overwritten, not accumulated)
 * Requires K % block == 0, N % 8 == 0, r % 8 == 0, r <= 64.
 * Errors as for qlora_linear_fwd. */
qlora_status qlora_linear_bwd(const qlora_nf4_weight *w, const uint16_t *x, const uint16_t *dY,
                              int64_t M, const uint16_t *A, const uint16_t *B, int32_t r,
                              float alpha, const float *t_saved, void *dX, qlora_dtype dx_dtype,
                              float *dA, float *dB, void *ws, size_t ws_bytes, uint32_t flags,
                              void *stream);

/* LoRA dropout on the bypass input.  [QLoRA-26] Step 5 training config and
 * [Gemma-9] LoraConfig (lora_dropout): in training the LoRA branch takes
 * dropout(x) = x . keep / (1 - p), keep ~ Bernoulli(1 - p) per element of
 * x, while the base branch takes x:
 *   y  = x . W_hat^T + s . (dropout(x) . A^T) . B^T          (s = alpha / r)
 *   t  = dropout(x) . A^T,  u = dY . B
 *   dX = dY . W_hat + s / (1 - p) . keep . (u . A)
 *   dA = s / (1 - p) . u^T . (x . keep),   dB = s . dY^T . t
 * `mask` holds the keep bits of the [M, K] input x as produced by
 * qlora_dropout_mask (device, caller-owned, const in the calls); p is the
 * probability it was drawn with (0 <= p < 1; 1/(1 - p) in fp32). */
typedef struct {
  const uint32_t *mask;
  float p;
} qlora_lora_dropout;

/* Words (uint32) per row of the keep mask of an [M, K] input:
 * ceil(K / 128) * 4 (a row is a whole number of 16-byte pieces).  Host only. */
qlora_status qlora_dropout_mask_words(int64_t K, int64_t *words_per_row);

/* Draw the keep mask of an [M, K] input (device, [M][words_per_row] uint32;
 * bit b of word w of row m is element k = 32 w + b; bits past K are 0).
 * The pages name no generator; this library uses the counter-based
 * Philox4x64-10 (Salmon et al., SC 2011) keyed by {seed, 0}: element
 * e = m K + k takes the 32-bit half (e mod 2, low half first) of 64-bit
 * output e / 2 of the stream, output o being word o mod 4 of the block at
 * counter {o / 4 + 1, 0, 0, 0}; it is kept when that uniform is at least
 * round(p 2^32).  Requires K % 64 == 0, 0 <= p < 1, mask 16-byte aligned.
 * Errors: QLORA_ERR_INVALID_ARG, QLORA_ERR_SHAPE, QLORA_ERR_ALIGN, QLORA_ERR_CUDA. */
qlora_status qlora_dropout_mask(uint64_t seed, float p, int64_t M, int64_t K, uint32_t *mask,
                                void *stream);

/* qlora_linear_fwd with LoRA dropout (dropout != NULL): the same arguments
 * and results, t_save receiving t = dropout(x) . A^T.  Both forward kernels
 * (GEMM and decode GEMV) take it. */
qlora_status qlora_linear_fwd_dropout(const qlora_nf4_weight *w, const uint16_t *x, int64_t M,
                                      const uint16_t *A, const uint16_t *B, int32_t r,
                                      float alpha, const qlora_lora_dropout *dropout, void *y,
                                      qlora_dtype y_dtype, float *t_save, void *ws,
                                      size_t ws_bytes, uint32_t flags, void *stream);

/* qlora_linear_bwd with LoRA dropout (dropout != NULL; the mask of the
 * forward).  dX is fp32: the dX GEMM seeds its accumulator with
 * s / (1 - p) . u . A at every position and a second kernel takes that term
 * back out where x was dropped. */
qlora_status qlora_linear_bwd_dropout(const qlora_nf4_weight *w, const uint16_t *x,
                                      const uint16_t *dY, int64_t M, const uint16_t *A,
                                      const uint16_t *B, int32_t r, float alpha,
                                      const qlora_lora_dropout *dropout, const float *t_saved,
                                      float *dX, float *dA, float *dB, void *ws, size_t ws_bytes,
                                      uint32_t flags, void *stream);

/* Backward without a caller workspace, for callers that cannot allocate
 * device memory (code that runs during CUDA graph capture, hosts whose
 * allocator forbids allocation on a hot path, or that give the library only
 * its inputs and outputs).  The pages have no counterpart: this is a
 * deployment convenience of this library.
 * Same arguments, results and errors as qlora_linear_bwd, minus ws and
 * ws_bytes.  Its workspace is a fixed array of QLORA_NOALLOC_SCRATCH_BYTES
 * in the library's device memory, held by every GPU that loads the library
 * until the process exits; the call allocates and frees nothing.
 *   - Sizes whose qlora_workspace_size_min exceeds
 *     QLORA_NOALLOC_SCRATCH_BYTES return QLORA_ERR_WORKSPACE (16 MiB covers
 *     the Llama-3-8B projection shapes at r = 16 up to 8192 tokens).  The
 *     array has no split-tile area, so the dX GEMM computes whole tiles.
 *   - The first call on a device looks up the array's device address (a
 *     CUDA runtime query, no allocation) and caches it; make that first call
 *     before any stream capture.
 *   - Every call on a device shares the one array, which keeps what the
 *     last call left in it.  The parts a call reads before writing (the
 *     device status word and the dA/dB tile counters, which must start at
 *     zero) are zeroed on `stream` at the start of each call (two memsets,
 *     no allocation), so calls of different sizes, or a call after one that
 *     timed out, start clean.  Calls that overlap on the GPU (different
 *     streams, no ordering between them) race on the array and give
 *     undefined results.
 *   - A device-side timeout is not reported by this entry point (it has no
 *     workspace the caller could read). */
#define QLORA_NOALLOC_SCRATCH_BYTES (16u << 20)
qlora_status qlora_linear_bwd_noalloc(const qlora_nf4_weight *w, const uint16_t *x,
                                      const uint16_t *dY, int64_t M, const uint16_t *A,
                                      const uint16_t *B, int32_t r, float alpha,
                                      const float *t_saved, void *dX, qlora_dtype dx_dtype,
                                      float *dA, float *dB, uint32_t flags, void *stream);

/* The 15 fp32 decision thresholds the quantiser uses with table `codebook`:
 * element index = number of thresholds <= (w / absmax).  Derived on the host
 * from the table and the nearest-codepoint rule above.  Host only, no GPU
 * needed.  QLORA_ERR_INVALID_ARG for an unknown codebook. */
qlora_status qlora_nf4_thresholds(int32_t codebook, float out[15]);

/* The 16 codepoints of table `codebook` as fp32 (see qlora_codebook).  Host
 * only.  QLORA_ERR_INVALID_ARG for an unknown codebook. */
qlora_status qlora_nf4_codebook(int32_t codebook, float out[16]);

const char *qlora_status_string(qlora_status s);

#ifdef __cplusplus
}
#endif

#endif /* QLORA_B300_H */
