// dropout.cu -- LoRA dropout on the bypass input, sm_103a.
//
// "QLoRA and 4bit Quantization | QLoRA 与 4-bit 量化", Step 5 training config
// and "第 09 期 | QLoRA 4-bit 量化微调" LoraConfig (lora_dropout = p): in
// training the LoRA branch sees dropout(x) = x . keep / (1 - p), keep ~
// Bernoulli(1 - p) per element; the base branch sees x.
//
// The keep mask of an [M, K] input is a bit matrix [M][words_per_row] of
// uint32 (bit b of word w of row m: element k = 32 w + b; words_per_row =
// ceil(K / 128) * 4, so that a row is a whole number of 16-byte pieces;
// bits past K are 0).  Element e = m K + k draws the 32-bit uniform
//   u = half (e mod 2) of output e / 2 of the Philox4x64-10 stream keyed by
//       {seed, 0}, output o being word o mod 4 of the block at counter
//       {o / 4 + 1, 0, 0, 0} (Salmon, Moraes, Dror and Shaw, "Parallel random
//       numbers: as easy as 1, 2, 3", SC 2011; 10 rounds, multipliers and
//       Weyl key increments of the published 4x64 variant),
// and is kept when u >= round(p 2^32).
//
// The mask is used by the LoRA down-projection (t), the t kernel of the
// decode path, and the dA contraction; the dX GEMM seeds its accumulator
// with the full s/(1-p) (u A) and dropout_dx_fix_kernel then takes the term
// back out at the dropped positions (fp32 dX).
#include "common.cuh"
#include "kernels.h"

namespace qlora {

__device__ __forceinline__ void philox4x64_10(uint64_t c[4], uint64_t k0, uint64_t k1) {
  const uint64_t M0 = 0xD2E7470EE14C6C93ull, M1 = 0xCA5A826395121157ull;
  const uint64_t W0 = 0x9E3779B97F4A7C15ull, W1 = 0xBB67AE8584CAA73Bull;
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += W0;
      k1 += W1;
    }
    const uint64_t hi0 = __umul64hi(M0, c[0]), lo0 = M0 * c[0];
    const uint64_t hi1 = __umul64hi(M1, c[2]), lo1 = M1 * c[2];
    const uint64_t n0 = hi1 ^ c[1] ^ k0, n2 = hi0 ^ c[3] ^ k1;
    c[0] = n0;
    c[1] = lo1;
    c[2] = n2;
    c[3] = lo0;
  }
}

// One thread per mask word: 32 consecutive elements of one row (K % 64 == 0,
// so a word never crosses a row) = 4 Philox blocks.
__global__ void __launch_bounds__(256) dropout_mask_kernel(uint64_t seed, uint32_t p32,
                                                           int64_t M, int K, int wpr,
                                                           uint32_t *__restrict__ mask) {
  pdl_wait_release();
  const int64_t total = M * wpr;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t m = i / wpr;
    const int w = (int)(i - m * wpr);
    uint32_t bits = 0;
    if (w * 32 < K) {
      const uint64_t e0 = (uint64_t)m * (uint64_t)K + (uint64_t)w * 32;  // multiple of 32
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        uint64_t c[4] = {e0 / 8 + 1 + b, 0, 0, 0};
        philox4x64_10(c, seed, 0);
#pragma unroll
        for (int o = 0; o < 4; ++o) {
          const uint32_t u0 = (uint32_t)c[o], u1 = (uint32_t)(c[o] >> 32);
          bits |= (uint32_t)(u0 >= p32) << (b * 8 + 2 * o);
          bits |= (uint32_t)(u1 >= p32) << (b * 8 + 2 * o + 1);
        }
      }
    }
    mask[i] = bits;
  }
}

cudaError_t launch_dropout_mask(uint64_t seed, uint32_t p32, int64_t M, int K, int wpr,
                                uint32_t *mask, int num_sms, cudaStream_t s) {
  if (M == 0) return cudaSuccess;
  const int64_t total = M * wpr;
  int64_t grid = (total + 255) / 256;
  if (grid > (int64_t)num_sms * 16) grid = (int64_t)num_sms * 16;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute at[1] = {pdl_attr()};
  cfg.attrs = at;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, dropout_mask_kernel, seed, p32, M, K, wpr, mask);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// dX[m, k] -= sum_j lb[m, j] At[k, j] at every dropped (m, k): the dX GEMM
// seeded its accumulator with exactly these bf16 operands for every (m, k).
// One thread per 8 columns of one row (one byte of a keep word): the row of lb
// and each dropped column's row of At are read with 16-byte loads.
template <int KS>  // KS = RP / 8 16-byte pieces per row
__global__ void __launch_bounds__(256) dropout_dx_fix_kernel(
    const uint32_t *__restrict__ mask, int wpr, int64_t M, int K,
    const uint16_t *__restrict__ lb, const uint16_t *__restrict__ At, float *__restrict__ dX) {
  pdl_wait_release();
  constexpr int RP = KS * 8;
  const int k8s = K >> 3;  // pieces of 8 columns per row (K % 64 == 0)
  const int64_t total = M * k8s;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t m = i / k8s;
    const int p8 = (int)(i - m * k8s);
    const uint32_t w = __ldg(mask + m * wpr + (p8 >> 2));
    uint32_t drop = ~(w >> ((p8 & 3) * 8)) & 0xffu;
    if (drop == 0u) continue;
    float um[RP];
    const uint4 *lr = reinterpret_cast<const uint4 *>(lb + m * RP);
#pragma unroll
    for (int q = 0; q < KS; ++q) {
      const uint4 v = __ldg(lr + q);
      um[8 * q + 0] = bf16_lo(v.x), um[8 * q + 1] = bf16_hi(v.x);
      um[8 * q + 2] = bf16_lo(v.y), um[8 * q + 3] = bf16_hi(v.y);
      um[8 * q + 4] = bf16_lo(v.z), um[8 * q + 5] = bf16_hi(v.z);
      um[8 * q + 6] = bf16_lo(v.w), um[8 * q + 7] = bf16_hi(v.w);
    }
    while (drop) {
      const int b = __ffs(drop) - 1;
      drop &= drop - 1;
      const int k = p8 * 8 + b;
      const uint4 *ak = reinterpret_cast<const uint4 *>(At + (int64_t)k * RP);
      float v = 0.f;
#pragma unroll
      for (int q = 0; q < KS; ++q) {
        const uint4 a = __ldg(ak + q);
        v = fmaf(um[8 * q + 0], bf16_lo(a.x), v);
        v = fmaf(um[8 * q + 1], bf16_hi(a.x), v);
        v = fmaf(um[8 * q + 2], bf16_lo(a.y), v);
        v = fmaf(um[8 * q + 3], bf16_hi(a.y), v);
        v = fmaf(um[8 * q + 4], bf16_lo(a.z), v);
        v = fmaf(um[8 * q + 5], bf16_hi(a.z), v);
        v = fmaf(um[8 * q + 6], bf16_lo(a.w), v);
        v = fmaf(um[8 * q + 7], bf16_hi(a.w), v);
      }
      dX[m * K + k] -= v;
    }
  }
}

cudaError_t launch_dropout_dx_fix(const uint32_t *mask, int wpr, int64_t M, int K,
                                  const uint16_t *lb, const uint16_t *At, int RP, float *dX,
                                  int num_sms, cudaStream_t s) {
  if (M == 0) return cudaSuccess;
  const int64_t total = M * (K / 8);
  int64_t grid = (total + 255) / 256;
  if (grid > (int64_t)num_sms * 16) grid = (int64_t)num_sms * 16;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute at[1] = {pdl_attr()};
  cfg.attrs = at;
  cfg.numAttrs = 1;
  switch (RP / 8) {
    case 2: return cudaLaunchKernelEx(&cfg, dropout_dx_fix_kernel<2>, mask, wpr, M, K, lb, At, dX);
    case 4: return cudaLaunchKernelEx(&cfg, dropout_dx_fix_kernel<4>, mask, wpr, M, K, lb, At, dX);
    case 6: return cudaLaunchKernelEx(&cfg, dropout_dx_fix_kernel<6>, mask, wpr, M, K, lb, At, dX);
    case 8: return cudaLaunchKernelEx(&cfg, dropout_dx_fix_kernel<8>, mask, wpr, M, K, lb, At, dX);
  }
  return cudaErrorInvalidValue;
}

}  // namespace qlora
