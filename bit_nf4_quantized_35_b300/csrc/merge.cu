// merge.cu -- adapter merge for sm_103a:
//   W_out[n, k] = bf16_rn( w_hat[n, k] + s . sum_j B[n, j] A[j, k] ),  s = alpha / r
// ("QLoRA and 4bit Quantization | QLoRA 与 4-bit 量化", Step 5 conclusion:
// the merged adapter is what deployment loads; the forward formula of Step 3
// gives x W_hat^T + s (x A^T) B^T = x (W_hat + s B A)^T).
//
// HBM-bound (0.5 packed + 2 output bytes per weight).  A warp takes a unit of
// 16 rows x 256 columns (4 blocks of 64); a CTA of 8 warps takes 8 row tiles
// of one 256-column chunk, so the chunk of A is staged once per CTA.
//   - w_hat: lane (g, tq) dequantises rows g and g+8 of block tq with the
//     per-block byte-permute table (the dequantiser's routine: exact bf16).
//   - B A: bf16 mma.sync m16n8k16 (fp32 accumulation), A-operand = 16 rows
//     of B, B-operand = A.  The columns of n-tile j are mapped to positions
//     2j, 2j+1 of each lane group's block (column c -> block c / 2, position
//     2j + c % 2), so a lane's accumulator holds exactly the positions whose
//     w_hat pair its table lookup produced.
//   - A chunk in shared memory as [256 columns][RP ranks] bf16 with the
//     ranks of a row interleaved (0 1 8 9 2 3 10 11 ...) so that a lane's two
//     B-operand words are one 8-byte load.
//   - epilogue: fp32 w_hat + s . (B A), one rounding to bf16, 16-byte stores.
#include "common.cuh"
#include "kernels.h"

namespace qlora {

constexpr int kMergeWarps = 8;

// A plain register function (no volatile), so that the compiler can
// interleave the MMAs with the loads and the table lookups.
__device__ __forceinline__ void mma_bf16_m(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                           uint32_t a3, uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Position of rank j inside an interleaved group of 16: 0 1 8 9 2 3 10 11 ...
__device__ __forceinline__ int rank_slot(int j) {
  const int q = j & 15;
  return (j & ~15) | (((q & 7) >> 1) << 2) | ((q >> 3) << 1) | (q & 1);
}

template <int KS>  // KS = RP / 16 rank steps
__global__ void __launch_bounds__(kMergeWarps * 32) merge_lora_kernel(const MergeArgs p) {
  __shared__ __align__(16) uint16_t as[256 * KS * 16];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tq = lane & 3;
  const int chunk = blockIdx.y;
  const int kc0 = chunk * 256;
  constexpr int RP = KS * 16;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // A chunk -> shared memory, transposed and rank-interleaved (0 past r or K)
  for (int i = threadIdx.x; i < 256 * RP; i += blockDim.x) {
    const int j = i / 256, c = i - j * 256;
    const int k = kc0 + c;
    uint16_t v = 0;
    if (j < p.r && k < p.K) v = p.A[(int64_t)j * p.K + k];
    as[c * RP + rank_slot(j)] = v;
  }
  __syncthreads();
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const int tile = blockIdx.x * kMergeWarps + warp;
  const int n0 = tile * 16 + g, n1 = n0 + 8;
  if (tile * 16 >= p.N) return;
  const int blk = chunk * 4 + tq;  // 64-chunk of the row
  const int kbr = p.K >> 6;
  const bool kin = blk < kbr;
  const bool ok0 = kin && n0 < p.N, ok1 = kin && n1 < p.N;
  // packed bytes and block constants of rows n0, n1, block blk
  auto fetch = [&](int n, bool ok, uint4 &lo, uint4 &hi, float &ahat) {
    lo = hi = make_uint4(0, 0, 0, 0);
    ahat = 0.f;
    if (!ok) return;
    const uint8_t *src = p.packed + ((int64_t)n * kbr + blk) * 32;
    lo = ldg_nc_v4(src);
    hi = ldg_nc_v4(src + 16);
    const int64_t b = ((int64_t)n * kbr + blk) >> p.bshift;
    const float cv = ldg_nc_f32(p.cvec + (b >> p.cshift));
    ahat = p.use_code ? __fmul_rn((float)ldg_nc_s8(p.codes + b), cv) : cv;
  };
  uint4 l0, h0, l1, h1;
  float ah0, ah1;
  fetch(n0, ok0, l0, h0, ah0);
  fetch(n1, ok1, l1, h1, ah1);
  // A-operand fragments: rows n0 / n1 of B, ranks 2tq, 2tq+1 (+8) of each 16-step
  uint32_t af[KS][4];
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    const int j0 = ks * 16 + 2 * tq;
    auto bw = [&](int n, int j) -> uint32_t {
      if (n >= p.N || j >= p.r) return 0u;
      return *reinterpret_cast<const uint32_t *>(p.B + (int64_t)n * p.r + j);
    };
    af[ks][0] = bw(n0, j0);
    af[ks][1] = bw(n1, j0);
    af[ks][2] = bw(n0, j0 + 8);
    af[ks][3] = bw(n1, j0 + 8);
  }
  const Nf4Table t0 = make_table(ah0, p.cb), t1 = make_table(ah1, p.cb);
  const uint32_t w0[8] = {l0.x, l0.y, l0.z, l0.w, h0.x, h0.y, h0.z, h0.w};
  const uint32_t w1[8] = {l1.x, l1.y, l1.z, l1.w, h1.x, h1.y, h1.z, h1.w};
  // this lane's column of every n-tile: block g >> 1, position 2j + (g & 1)
  const int bcol = (g >> 1) * 64 + (g & 1);
  uint16_t *out0 = p.out + (int64_t)n0 * p.K + (int64_t)blk * 64;
  uint16_t *out1 = p.out + (int64_t)n1 * p.K + (int64_t)blk * 64;
#pragma unroll
  for (int wi = 0; wi < 8; ++wi) {
    uint32_t o0[4], o1[4];
    lookup8(t0, w0[wi], o0);
    lookup8(t1, w1[wi], o1);
    uint32_t r0[4], r1[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int j = wi * 4 + q;  // n-tile: positions 2j, 2j + 1
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      const uint2 *arow = reinterpret_cast<const uint2 *>(as + (bcol + 2 * j) * RP + tq * 4);
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const uint2 bv = arow[ks * 4];  // 16 ranks = 32 bytes = 4 uint2 per step
        mma_bf16_m(d, af[ks][0], af[ks][1], af[ks][2], af[ks][3], bv.x, bv.y);
      }
      r0[q] = pack_bf16x2(fmaf(p.s, d[0], bf16_lo(o0[q])), fmaf(p.s, d[1], bf16_hi(o0[q])));
      r1[q] = pack_bf16x2(fmaf(p.s, d[2], bf16_lo(o1[q])), fmaf(p.s, d[3], bf16_hi(o1[q])));
    }
    if (ok0) *reinterpret_cast<uint4 *>(out0 + wi * 8) = make_uint4(r0[0], r0[1], r0[2], r0[3]);
    if (ok1) *reinterpret_cast<uint4 *>(out1 + wi * 8) = make_uint4(r1[0], r1[1], r1[2], r1[3]);
  }
}

cudaError_t launch_merge(const MergeArgs &a, cudaStream_t s) {
  if (a.N == 0 || a.K == 0) return cudaSuccess;
  const int tiles = (a.N + 15) / 16;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((tiles + kMergeWarps - 1) / kMergeWarps, (a.K + 255) / 256, 1);
  cfg.blockDim = dim3(kMergeWarps * 32, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute at[1] = {pdl_attr()};
  cfg.attrs = at;
  cfg.numAttrs = 1;
  const int ks = (a.r + 15) / 16;
  switch (ks) {
    case 1: return cudaLaunchKernelEx(&cfg, merge_lora_kernel<1>, a);
    case 2: return cudaLaunchKernelEx(&cfg, merge_lora_kernel<2>, a);
    case 3: return cudaLaunchKernelEx(&cfg, merge_lora_kernel<3>, a);
    case 4: return cudaLaunchKernelEx(&cfg, merge_lora_kernel<4>, a);
  }
  return cudaErrorInvalidValue;
}

}  // namespace qlora
