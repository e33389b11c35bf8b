// kernels.h -- internal declarations shared by the kernel files and the C ABI
// implementation (argument structs and host-side launchers).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace qlora {

// Fused dequantise + tcgen05 GEMM (gemm_tc.cu).
struct GemmArgs {
  const uint8_t *packed;
  const int8_t *codes;
  const float *absf;
  const float *scale2;
  int group;
  int64_t wrows;  // N
  int64_t wcols;  // K
  int M;
  int out_cols;   // N (forward) or K (dX)
  int kdim;       // contraction length: K (forward) or N (dX)
  int r;
  int r_pad;
  float s;
  void *out;
  int out_bf16;
  int stages;
  int *status;
  // Branch-free block constant: a_hat = use_code ? code[b] * cvec[b / cdiv] : cvec[b / cdiv]
  // (set by the launcher; `codes` points at readable memory even without DQ).
  const float *cvec;
  int cdiv;
  int use_code;
  int cshift;  // log2(cdiv): cdiv is 1 or a power of two
  int bshift;  // log2(block / 64): a 64-element chunk c lies in block c >> bshift
  int bn;      // output columns per CTA pair: 128..256, multiple of 32 (set by the launcher)
  // Split tiles (stream-K).  With sk_part set, each cluster takes an equal
  // share of the (tile, 64-wide contraction block) units and a tile shared by
  // several clusters is summed from fp32 partials by the last one to finish.
  // sk_part: 2 * sk_slots_clusters * 2 * 128 * 256 floats; sk_count:
  // 2 * sk_slots_clusters ints, zero between calls.  Null: whole tiles only.
  float *sk_part;
  int *sk_count;
  int sk_slots_clusters;
  int sk;        // 1 when this launch splits tiles (from gemm_plan)
  int clusters;  // CTA pairs launched (from gemm_plan)
  Codebook cb;   // the 16 codepoints of the weight's table
};
// Launch shape of the fused GEMM for one call: pair-tile width, split mode
// and cluster count.  sk_slots_clusters = 0 means no split-tile area.
struct GemmPlan {
  int bn, sk, clusters;
};
cudaError_t gemm_plan(bool dx, int M, int out_cols, int kdim, int r_pad, int sk_slots_clusters,
                      GemmPlan *plan);
// Upper bound on the clusters any launch uses on the current device (sizes
// the split-tile area).
int gemm_cluster_bound();
cudaError_t launch_gemm(bool dx, const CUtensorMap &tmA, const CUtensorMap &tmL1,
                        const CUtensorMap &tmL2, const GemmArgs &args, cudaStream_t s);
int gemm_pick_stages(int r_pad);

// Decode GEMV (gemv.cu): t kernel + weight-streaming kernel.
struct GemvArgs {
  const uint8_t *packed;
  const int8_t *codes;  // readable memory even without DQ (use_code = 0)
  const float *cvec;    // s2 (DQ) or fp32 absmax: a_hat = use_code ? code[b] * cvec[b >> cshift] : cvec[b]
  int use_code, cshift, bshift;
  int N, K;
  const uint16_t *x;  // [M, K] bf16
  int M;
  const uint16_t *B;  // [N, r] bf16
  int r, RP;
  float s;
  void *y;
  int y_bf16;
  const float *t;  // [M, RP] fp32 in the workspace, written by the t kernel
  int *status;     // device status word
  const uint32_t *mask;  // LoRA dropout keep bits of x ([M][wpr]) or null
  int wpr;
  float keep_scale;
  // set by the launcher from the plan:
  int S, slice_chunks, clusters, tiles_total, tiles_max, depth;
  Codebook cb;
};
// Launch shape of the decode GEMV: S CTAs per cluster (K slices of
// slice_chunks x 256 columns), clusters owning ranges of 16-row tiles.
struct GemvPlan {
  int S, slice_chunks, clusters, tiles_total, tiles_max, smem, depth;
};
// 0 when the decode kernel takes this shape on num_sms SMs (plan filled), else -1.
int gemv_plan(int N, int K, int M, int r, int num_sms, GemvPlan *plan);
// tmW: 2-D uint8 tensor map of the packed weight [N, K/2], box 128 x 16,
// 128-byte swizzle.  tpart: ceil(K/256) x M x RP floats of scratch; counter:
// one int, zero before the call and after it.
cudaError_t launch_gemv(const CUtensorMap &tmW, GemvArgs a, const GemvPlan &plan,
                        const uint16_t *A, float *tpart, int *counter, float *t_save,
                        cudaStream_t s);
// out[m, j] = sum_c G[m, c] H[j, c] (fp32, j < r) and outb[m, j] = bf16(s . out[m, j])
// (j < r_pad, zero beyond r); either output may be null.  H has r rows of C.
// With `mask` (LoRA dropout keep bits of G, wpr words per row) the dropped
// elements of G are zeroed and out = keep_scale . G H^T, outb = bf16(s . out).
cudaError_t launch_lora_down(const uint16_t *G, int64_t M, int C, const uint16_t *H, int r,
                             float s, float *out, uint16_t *outb, int r_pad, int num_sms,
                             cudaStream_t st, const uint32_t *mask = nullptr, int wpr = 0,
                             float keep_scale = 1.0f);
// The same for wide inputs (C >= 8192), from TMA tensor maps: tmG of G [M, C]
// (box 64 x 16), tmH of H [r, C] (box 64 x r_pad8, r_pad8 = 8 . an even number
// of 8-row tiles >= r), both in the 128-byte swizzle.  status: the device
// status word (its waits are bounded).
cudaError_t launch_lora_down_tma(const CUtensorMap &tmG, const CUtensorMap &tmH, int64_t M,
                                 int C, int r, float s, float *out, uint16_t *outb, int r_pad,
                                 int num_sms, int *status, cudaStream_t st,
                                 const uint32_t *mask = nullptr, int wpr = 0,
                                 float keep_scale = 1.0f);

// Quantise / dequantise (quantize.cu).
cudaError_t launch_quantize(const void *W, bool bf16_in, int block, int64_t nblocks, int group,
                            uint8_t *packed, int8_t *codes, float *absf, float *scale2,
                            int *nonfinite_flag, const float th[15], int num_sms,
                            cudaStream_t s);
cudaError_t launch_dequant(const uint8_t *packed, const int8_t *codes, const float *absf,
                           const float *scale2, int group, int block, int64_t nblocks,
                           uint16_t *out, const Codebook &cb, int num_sms, cudaStream_t s);

// Adapter merge (merge.cu): out = bf16(w_hat + s . B A).
struct MergeArgs {
  const uint8_t *packed;
  const int8_t *codes;  // readable memory even without DQ
  const float *cvec;
  int use_code, cshift, bshift;
  int N, K;
  const uint16_t *A;  // [r, K] bf16
  const uint16_t *B;  // [N, r] bf16
  int r;
  float s;
  uint16_t *out;  // [N, K] bf16
  Codebook cb;
  uint32_t k31, k16;  // 2^31 and 2^16 (multipliers of lookup8_mulhi)
};
// tmO: 3-D bf16 tensor map of `out` viewed as [N][K / 64][64], box 64 x 4 x 16,
// 128-byte swizzle (see qlora_merge_lora).
cudaError_t launch_merge(const CUtensorMap &tmO, const MergeArgs &a, int num_sms,
                         cudaStream_t s);

// Rank-r gradient contractions and layout helpers (lora_grad.cu).
int skinny_splits(int64_t M, int C, int budget = 296);
void skinny_splits_pair(int64_t M, int N, int K, int *sn, int *sk);
int skinny_tiles(int C);
// dst = sc . G^T V for G [M, C] bf16, V [M, r] fp32: dst[c * r + j], or
// dst[j * C + c] with transpose.  part: splits * C * RP floats of scratch;
// tile_count: skinny_tiles(C) ints, zero before the call and after it.
// One contraction dst = sc . G^T V of the dA / dB kernel (see launch_skinny).
struct SkinnyJob {
  const uint16_t *G;
  int C;
  const float *V;
  int64_t rows_per_split;
  int splits, tiles;
  float *part;      // splits * C * RP floats of scratch
  int *tile_count;  // tiles ints, zero before and after
  float sc;
  int transpose;
  float *dst;
  const uint32_t *mask;  // dropout keep bits of G or null
  int wpr;
};
SkinnyJob skinny_job(const uint16_t *G, int64_t M, int C, const float *V, float *part,
                     int *tile_count, int splits, float sc, bool transpose, float *dst,
                     const uint32_t *mask, int wpr);
// Two independent contractions over the same M rows in one launch (their
// part and tile_count areas must not overlap).
cudaError_t launch_skinny2(const SkinnyJob &j0, const SkinnyJob &j1, int64_t M, int r, int RP,
                           cudaStream_t s);
// With `mask` (dropout keep bits of G, wpr words per row) the dropped
// elements of G count as zero.
cudaError_t launch_skinny(const uint16_t *G, int64_t M, int C, const float *V, int r, int RP,
                          float *part, int *tile_count, int splits, float sc, bool transpose,
                          float *dst, cudaStream_t s, const uint32_t *mask = nullptr,
                          int wpr = 0);

// LoRA dropout (dropout.cu).  Keep bits [M][wpr] uint32 of an [M, K] input.
cudaError_t launch_dropout_mask(uint64_t seed, uint32_t p32, int64_t M, int K, int wpr,
                                uint32_t *mask, int num_sms, cudaStream_t s);
// dX[m, k] -= sum_j lb[m, j] At[k, j] (bf16 operands, fp32) at every dropped (m, k).
cudaError_t launch_dropout_dx_fix(const uint32_t *mask, int wpr, int64_t M, int K,
                                  const uint16_t *lb, const uint16_t *At, int RP, float *dX,
                                  int num_sms, cudaStream_t s);
cudaError_t launch_transposes(const uint16_t *A, const uint16_t *B, int N, int K, int r, int RP,
                              uint16_t *At, uint16_t *Bt, int num_sms, cudaStream_t s);

// Byte range [*off, *off + *bytes) of a (M, N, K, r) workspace holding the
// dA/dB column-tile counters, which must be zero when a backward call starts
// (capi.cu).  The device status word is the first 256 bytes.
void ws_counter_range(int64_t M, int64_t N, int64_t K, int r, size_t *off, size_t *bytes);

}  // namespace qlora
