// lora_grad.cu -- the rank-r gradient contractions of the QLoRA backward pass
// and small layout helpers, sm_103a.
//
// "QLoRA and 4bit Quantization | QLoRA 与 4-bit 量化", Step 3/4 (gradients
// reach lora_A and lora_B; the NF4 state gets none):
//   dB = s . dY^T . t     [N, r]   (t = x A^T from the forward, fp32)
//   dA = s . u^T  . x     [r, K]   (u = dY B from the dX GEMM, fp32)
// Both are "tall-skinny" products G^T V with G a bf16 [M, C] activation
// (dY or x) and V an fp32 [M, r] factor, reduced over the M tokens.  They
// run on the CUDA cores in fp32: the gradients are large sums (|dA|, |dB| of
// order 10^2 at M = 8192) that must keep ~1e-4 relative accuracy, which a
// bf16 operand V could not give.  Each thread owns two adjacent columns of G
// and all r_pad accumulators; V rows are staged in shared memory and read as
// broadcasts; the M range is split across CTAs and the partial sums are
// reduced in a fixed order by a second kernel (deterministic).
#include "common.cuh"
#include "kernels.h"

namespace qlora {

constexpr int kSkinnyThreads = 128;
constexpr int kSkinnyCols = 2 * kSkinnyThreads;  // columns per CTA
constexpr int kSkinnyRows = 64;                  // V rows staged per pass

template <int RP>
__global__ void __launch_bounds__(kSkinnyThreads) skinny_tn_kernel(
    const uint16_t *__restrict__ G, int64_t M, int C, const float *__restrict__ V, int r,
    int64_t rows_per_split, float *__restrict__ part) {
  __shared__ __align__(16) float vs[kSkinnyRows][RP];
  const int c = blockIdx.x * kSkinnyCols + threadIdx.x * 2;
  const bool cvalid = c < C;
  const int64_t m_lo = (int64_t)blockIdx.y * rows_per_split;
  int64_t m_hi = m_lo + rows_per_split;
  if (m_hi > M) m_hi = M;
  float a0[RP], a1[RP];
#pragma unroll
  for (int j = 0; j < RP; ++j) a0[j] = a1[j] = 0.f;
  for (int64_t mb = m_lo; mb < m_hi; mb += kSkinnyRows) {
    const int rows = (int)((m_hi - mb) < kSkinnyRows ? (m_hi - mb) : kSkinnyRows);
    __syncthreads();
    for (int i = threadIdx.x; i < kSkinnyRows * RP; i += kSkinnyThreads) {
      const int mm = i / RP, j = i % RP;
      vs[mm][j] = (mm < rows && j < r) ? V[(mb + mm) * r + j] : 0.f;
    }
    __syncthreads();
    const uint16_t *gp = G + mb * C + c;
    int mm = 0;
    for (; mm + 8 <= rows; mm += 8) {
      uint32_t gv[8];
#pragma unroll
      for (int q = 0; q < 8; ++q)
        gv[q] = cvalid ? __ldg(reinterpret_cast<const uint32_t *>(gp + (int64_t)(mm + q) * C)) : 0u;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float g0 = bf16_lo(gv[q]), g1 = bf16_hi(gv[q]);
        const float4 *vr = reinterpret_cast<const float4 *>(&vs[mm + q][0]);
#pragma unroll
        for (int j4 = 0; j4 < RP / 4; ++j4) {
          const float4 v = vr[j4];
          a0[4 * j4 + 0] = fmaf(g0, v.x, a0[4 * j4 + 0]);
          a0[4 * j4 + 1] = fmaf(g0, v.y, a0[4 * j4 + 1]);
          a0[4 * j4 + 2] = fmaf(g0, v.z, a0[4 * j4 + 2]);
          a0[4 * j4 + 3] = fmaf(g0, v.w, a0[4 * j4 + 3]);
          a1[4 * j4 + 0] = fmaf(g1, v.x, a1[4 * j4 + 0]);
          a1[4 * j4 + 1] = fmaf(g1, v.y, a1[4 * j4 + 1]);
          a1[4 * j4 + 2] = fmaf(g1, v.z, a1[4 * j4 + 2]);
          a1[4 * j4 + 3] = fmaf(g1, v.w, a1[4 * j4 + 3]);
        }
      }
    }
    for (; mm < rows; ++mm) {
      const uint32_t gv =
          cvalid ? __ldg(reinterpret_cast<const uint32_t *>(gp + (int64_t)mm * C)) : 0u;
      const float g0 = bf16_lo(gv), g1 = bf16_hi(gv);
#pragma unroll
      for (int j = 0; j < RP; ++j) {
        a0[j] = fmaf(g0, vs[mm][j], a0[j]);
        a1[j] = fmaf(g1, vs[mm][j], a1[j]);
      }
    }
  }
  if (cvalid) {
    float4 *d0 = reinterpret_cast<float4 *>(part + ((int64_t)blockIdx.y * C + c) * RP);
    float4 *d1 = d0 + RP / 4;
#pragma unroll
    for (int j4 = 0; j4 < RP / 4; ++j4) {
      d0[j4] = make_float4(a0[4 * j4], a0[4 * j4 + 1], a0[4 * j4 + 2], a0[4 * j4 + 3]);
      d1[j4] = make_float4(a1[4 * j4], a1[4 * j4 + 1], a1[4 * j4 + 2], a1[4 * j4 + 3]);
    }
  }
}

// dst = s * sum over splits (fixed order) of part[split][c][j], j < r.
// transpose == 0: dst[c * r + j] (dB layout [N, r]);
// transpose == 1: dst[j * C + c] (dA layout [r, K]).
__global__ void __launch_bounds__(256) reduce_parts_kernel(const float *__restrict__ part,
                                                           int splits, int C, int RP, int r,
                                                           float s, int transpose,
                                                           float *__restrict__ dst) {
  const int64_t total = (int64_t)C * r;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    int c, j;
    if (transpose) {
      j = (int)(i / C);
      c = (int)(i % C);
    } else {
      c = (int)(i / r);
      j = (int)(i % r);
    }
    float v = 0.f;
    for (int sp = 0; sp < splits; ++sp) v += part[((int64_t)sp * C + c) * RP + j];
    dst[i] = s * v;
  }
}

// Bt[j][n] = B[n][j] (j < r), 0 for r <= j < RP.
__global__ void transpose_b_kernel(const uint16_t *__restrict__ B, int N, int r, int RP,
                                   uint16_t *__restrict__ Bt) {
  const int64_t total = (int64_t)RP * N;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int j = (int)(i / N), n = (int)(i % N);
    Bt[i] = j < r ? B[(int64_t)n * r + j] : (uint16_t)0;
  }
}

// At[k][j] = A[j][k] (j < r), 0 for r <= j < RP.
__global__ void transpose_a_kernel(const uint16_t *__restrict__ A, int K, int r, int RP,
                                   uint16_t *__restrict__ At) {
  const int64_t total = (int64_t)K * RP;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int k = (int)(i / RP), j = (int)(i % RP);
    At[i] = j < r ? A[(int64_t)j * K + k] : (uint16_t)0;
  }
}

// ---------------------------------------------------------------------------
// LoRA down-projection out = G . H^T for a tall, skinny product:
//   forward  t = x . A^T   (G = x [M, K],  H = A  [r, K])
//   backward u = dY . B    (G = dY [M, N], H = B^T [r, N])
// It also writes bf16(s . out), zero-padded to r_pad columns: the operand of
// the rank-r MMAs that seed the fused GEMM's accumulator.
// One CTA per 16 rows of G, 8 warps splitting C; bf16 mma.sync m16n8k16 with
// fp32 accumulation (G streams from memory once, H is a few KB and stays in
// L1); the 8 warp partials meet in shared memory in a fixed order.
// Lane (g, q) loads 8 consecutive elements (16 B) of rows g and g+8 per 32
// columns; the two MMAs of those 32 columns pair their k indices in the same
// order for G and H, so any consistent assignment is exact.
constexpr int kDownWarps = 8;

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <int NT>  // n8 tiles: r_pad / 8
__global__ void __launch_bounds__(kDownWarps * 32) lora_down_kernel(
    const uint16_t *__restrict__ G, int64_t M, int C, const uint16_t *__restrict__ H, int r,
    float s, float *__restrict__ out, uint16_t *__restrict__ outb, int r_pad) {
  __shared__ float red[kDownWarps][16][NT * 8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;
  const int64_t m0 = (int64_t)blockIdx.x * 16;
  const int64_t rg = m0 + g, rg8 = m0 + g + 8;
  const bool vg = rg < M, vg8 = rg8 < M;
  // this warp's share of C, in 32-column chunks
  const int nch = (C + 31) / 32;
  const int per = (nch + kDownWarps - 1) / kDownWarps;
  const int c_lo = warp * per * 32;
  const int c_hi = min(C, (warp + 1) * per * 32);
  float d[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) d[nt][0] = d[nt][1] = d[nt][2] = d[nt][3] = 0.f;
  const uint16_t *g0p = G + (vg ? rg : 0) * C;
  const uint16_t *g8p = G + (vg8 ? rg8 : 0) * C;
  for (int c0 = c_lo; c0 < c_hi; c0 += 32) {
    const int cc = c0 + q * 8;
    const bool cv = cc < C;  // C % 8 == 0
    const uint4 a = ldg_nc_v4(g0p + (cv ? cc : 0));
    const uint4 b = ldg_nc_v4(g8p + (cv ? cc : 0));
    const uint32_t A0[4] = {vg && cv ? a.x : 0u, vg && cv ? a.y : 0u, vg && cv ? a.z : 0u,
                            vg && cv ? a.w : 0u};
    const uint32_t A8[4] = {vg8 && cv ? b.x : 0u, vg8 && cv ? b.y : 0u, vg8 && cv ? b.z : 0u,
                            vg8 && cv ? b.w : 0u};
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int j = nt * 8 + g;
      uint4 h = make_uint4(0, 0, 0, 0);
      if (j < r && cv) h = ldg_nc_v4(H + (int64_t)j * C + cc);
      // MMA 0: physical columns cc+0..3, MMA 1: cc+4..7
      mma_bf16_16816(d[nt], A0[0], A8[0], A0[1], A8[1], h.x, h.y);
      mma_bf16_16816(d[nt], A0[2], A8[2], A0[3], A8[3], h.z, h.w);
    }
  }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    red[warp][g][nt * 8 + 2 * q] = d[nt][0];
    red[warp][g][nt * 8 + 2 * q + 1] = d[nt][1];
    red[warp][g + 8][nt * 8 + 2 * q] = d[nt][2];
    red[warp][g + 8][nt * 8 + 2 * q + 1] = d[nt][3];
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 16 * NT * 8; i += blockDim.x) {
    const int row = i / (NT * 8), j = i % (NT * 8);
    const int64_t m = m0 + row;
    if (m >= M) continue;
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kDownWarps; ++w) v += red[w][row][j];
    if (out && j < r) out[m * r + j] = v;
    if (outb && j < r_pad)
      outb[m * r_pad + j] = j < r ? __bfloat16_as_ushort(__float2bfloat16_rn(s * v)) : (uint16_t)0;
  }
}

// ------------------------------------------------------------ launchers
cudaError_t launch_lora_down(const uint16_t *G, int64_t M, int C, const uint16_t *H, int r,
                             float s, float *out, uint16_t *outb, int r_pad, int num_sms,
                             cudaStream_t st) {
  (void)num_sms;
  if (M == 0) return cudaSuccess;
  const unsigned grid = (unsigned)((M + 15) / 16);
  switch ((r + 7) / 8) {
    case 1: lora_down_kernel<2><<<grid, kDownWarps * 32, 0, st>>>(G, M, C, H, r, s, out, outb, r_pad); break;
    case 2: lora_down_kernel<2><<<grid, kDownWarps * 32, 0, st>>>(G, M, C, H, r, s, out, outb, r_pad); break;
    case 3: lora_down_kernel<4><<<grid, kDownWarps * 32, 0, st>>>(G, M, C, H, r, s, out, outb, r_pad); break;
    case 4: lora_down_kernel<4><<<grid, kDownWarps * 32, 0, st>>>(G, M, C, H, r, s, out, outb, r_pad); break;
    case 5: lora_down_kernel<6><<<grid, kDownWarps * 32, 0, st>>>(G, M, C, H, r, s, out, outb, r_pad); break;
    case 6: lora_down_kernel<6><<<grid, kDownWarps * 32, 0, st>>>(G, M, C, H, r, s, out, outb, r_pad); break;
    case 7: lora_down_kernel<8><<<grid, kDownWarps * 32, 0, st>>>(G, M, C, H, r, s, out, outb, r_pad); break;
    case 8: lora_down_kernel<8><<<grid, kDownWarps * 32, 0, st>>>(G, M, C, H, r, s, out, outb, r_pad); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

int skinny_splits(int64_t M, int C) {
  const int coltiles = (C + kSkinnyCols - 1) / kSkinnyCols;
  int64_t sp = (296 + coltiles - 1) / coltiles;
  int64_t maxsp = M / 64;
  if (maxsp < 1) maxsp = 1;
  if (sp > maxsp) sp = maxsp;
  if (sp < 1) sp = 1;
  return (int)sp;
}

cudaError_t launch_skinny(const uint16_t *G, int64_t M, int C, const float *V, int r, int RP,
                          float *part, int splits, cudaStream_t s) {
  const int64_t rps = (M + splits - 1) / splits;
  dim3 grid((C + kSkinnyCols - 1) / kSkinnyCols, splits);
  switch (RP) {
    case 16: skinny_tn_kernel<16><<<grid, kSkinnyThreads, 0, s>>>(G, M, C, V, r, rps, part); break;
    case 32: skinny_tn_kernel<32><<<grid, kSkinnyThreads, 0, s>>>(G, M, C, V, r, rps, part); break;
    case 48: skinny_tn_kernel<48><<<grid, kSkinnyThreads, 0, s>>>(G, M, C, V, r, rps, part); break;
    case 64: skinny_tn_kernel<64><<<grid, kSkinnyThreads, 0, s>>>(G, M, C, V, r, rps, part); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_reduce_parts(const float *part, int splits, int C, int RP, int r, float sc,
                                bool transpose, float *dst, int num_sms, cudaStream_t s) {
  const int64_t total = (int64_t)C * r;
  int64_t blocks = (total + 255) / 256;
  if (blocks > (int64_t)num_sms * 8) blocks = (int64_t)num_sms * 8;
  if (blocks < 1) blocks = 1;
  reduce_parts_kernel<<<(unsigned)blocks, 256, 0, s>>>(part, splits, C, RP, r, sc,
                                                       transpose ? 1 : 0, dst);
  return cudaGetLastError();
}

cudaError_t launch_transposes(const uint16_t *A, const uint16_t *B, int N, int K, int r, int RP,
                              uint16_t *At, uint16_t *Bt, int num_sms, cudaStream_t s) {
  const int64_t tb = (int64_t)RP * N, ta = (int64_t)K * RP;
  int64_t gb = (tb + 255) / 256, ga = (ta + 255) / 256;
  const int64_t cap = (int64_t)num_sms * 8;
  if (gb > cap) gb = cap;
  if (ga > cap) ga = cap;
  transpose_b_kernel<<<(unsigned)gb, 256, 0, s>>>(B, N, r, RP, Bt);
  transpose_a_kernel<<<(unsigned)ga, 256, 0, s>>>(A, K, r, RP, At);
  return cudaGetLastError();
}

}  // namespace qlora
