// lora_grad.cu -- the rank-r gradient contractions of the QLoRA backward pass
// and small layout helpers, sm_103a.
//
// "QLoRA and 4bit Quantization | QLoRA 与 4-bit 量化", Step 3/4 (gradients
// reach lora_A and lora_B; the NF4 state gets none):
//   dB = s . dY^T . t     [N, r]   (t = x A^T from the forward, fp32)
//   dA = s . u^T  . x     [r, K]   (u = dY B from the backward pre-pass, fp32)
// Both are "tall-skinny" products G^T V with G a bf16 [M, C] activation
// (dY or x) and V an fp32 [M, r] factor, reduced over the M tokens.  The
// gradients are large sums (|dA|, |dB| of order 10^2 at M = 8192) that must
// keep ~1e-4 relative accuracy, which a bf16 V could not give: V is split
// exactly into bf16 hi + lo parts (16 significant bits) and both halves run
// through bf16 tensor-core MMAs with fp32 accumulation.  The M range is split
// across CTAs and the partial sums are reduced in a fixed order by a second
// kernel (deterministic).
#include "common.cuh"
#include "kernels.h"

namespace qlora {

// ---------------------------------------------------------------------------
// part[split][c][j] = sum_{m in split} G[m][c] . V[m][j]   (j < r_pad)
// One CTA = 128 columns c x one M split, 8 warps of 16 columns each.  Per
// 64-row chunk of M: the G tile [64 m][128 c] arrives by cp.async (double
// buffered, rows padded to 272 B so ldmatrix rows hit distinct banks) and
// V^T as bf16 hi and lo rows [2 r_pad][64 m] (padded to 144 B).  The MMA
// A operand (16 c x 16 m) is an ldmatrix.trans of the G tile, the B operand
// (16 m x 8 j) an ldmatrix of V^T.
constexpr int kGradThreads = 256;
constexpr int kGradCols = 128;  // c per CTA
constexpr int kGradRows = 64;   // m per chunk
constexpr int kGsPitch = 136;   // halves per G-tile row (128 + 8)
constexpr int kVtPitch = 72;    // halves per V^T row (64 + 8)

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

__host__ __device__ inline int grad_smem_bytes(int RPAD) {
  return 2 * kGradRows * kGsPitch * 2 + 2 * (2 * RPAD) * kVtPitch * 2;
}

template <int RPT>  // r_pad / 8
__global__ void __launch_bounds__(kGradThreads) lora_grad_tc_kernel(
    const uint16_t *__restrict__ G, int64_t M, int C, const float *__restrict__ V, int r,
    int64_t rows_per_split, float *__restrict__ part) {
  constexpr int RPAD = RPT * 8;
  constexpr int NJ = 2 * RPAD;  // hi rows then lo rows
  constexpr int NTT = NJ / 8;   // n8 tiles
  extern __shared__ __align__(16) uint16_t gsm[];
  uint16_t *gs = gsm;                                 // [2][64][136]
  uint16_t *vt = gsm + 2 * kGradRows * kGsPitch;      // [2][NJ][72]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;
  const int c0 = blockIdx.x * kGradCols;
  const int64_t m_lo = (int64_t)blockIdx.y * rows_per_split;
  const int64_t m_hi = min(M, m_lo + rows_per_split);
  const int nchunks = (int)((m_hi - m_lo + kGradRows - 1) / kGradRows);

  auto issue_g = [&](int ch, int buf) {  // 64 x 128 bf16 = 1024 16-byte pieces
    const int64_t mb = m_lo + (int64_t)ch * kGradRows;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = threadIdx.x + u * kGradThreads;
      const int row = i >> 4, cc = (i & 15) * 8;
      const int64_t m = mb + row;
      const int c = c0 + cc;
      const bool ok = m < m_hi && c < C;
      const uint16_t *src = G + (ok ? m * C + c : 0);
      cp_async16(smem_u32(gs + (buf * kGradRows + row) * kGsPitch + cc), src, ok ? 16u : 0u);
    }
    cp_async_commit();
  };
  auto stage_v = [&](int ch, int buf) {  // V rows -> bf16 hi / lo, transposed
    const int64_t mb = m_lo + (int64_t)ch * kGradRows;
    for (int i = threadIdx.x; i < kGradRows * RPAD; i += kGradThreads) {
      const int row = i / RPAD, j = i % RPAD;
      const int64_t m = mb + row;
      const float v = (m < m_hi && j < r) ? V[m * r + j] : 0.f;
      const __nv_bfloat16 hi = __float2bfloat16_rn(v);
      const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
      vt[(buf * NJ + j) * kVtPitch + row] = __bfloat16_as_ushort(hi);
      vt[(buf * NJ + RPAD + j) * kVtPitch + row] = __bfloat16_as_ushort(lo);
    }
  };

  float d[NTT][4];
#pragma unroll
  for (int nt = 0; nt < NTT; ++nt) d[nt][0] = d[nt][1] = d[nt][2] = d[nt][3] = 0.f;
  if (nchunks > 0) {
    issue_g(0, 0);
    stage_v(0, 0);
    cp_async_wait_all();
    __syncthreads();
  }
  const int cw = warp * 16;  // this warp's 16 columns inside the tile
  // ldmatrix lane roles: matrix mi = lane >> 3, row within it lane & 7
  const int mi = lane >> 3, lr = lane & 7;
  for (int ch = 0; ch < nchunks; ++ch) {
    const int cur = ch & 1;
    if (ch + 1 < nchunks) issue_g(ch + 1, cur ^ 1);
#pragma unroll
    for (int kk = 0; kk < kGradRows / 16; ++kk) {
      const int m0 = kk * 16;
      // A = G^T (16 c x 16 m): matrices (m0.., cw), (m0.., cw+8), (m0+8.., cw), (m0+8.., cw+8)
      uint32_t a0, a1, a2, a3;
      {
        const int row = m0 + lr + ((mi >> 1) << 3);
        const int col = cw + ((mi & 1) << 3);
        ldsm_x4_t(smem_u32(gs + (cur * kGradRows + row) * kGsPitch + col), a0, a1, a2, a3);
      }
#pragma unroll
      for (int np = 0; np < NTT / 2; ++np) {
        // B = V^T rows (j') x m: matrices (rows 16np.., m0), (16np.., m0+8),
        // (16np+8.., m0), (16np+8.., m0+8)
        uint32_t b0, b1, b2, b3;
        const int row = np * 16 + lr + ((mi >> 1) << 3);
        const int col = m0 + ((mi & 1) << 3);
        ldsm_x4(smem_u32(vt + (cur * NJ + row) * kVtPitch + col), b0, b1, b2, b3);
        mma_bf16_16816(d[2 * np], a0, a1, a2, a3, b0, b1);
        mma_bf16_16816(d[2 * np + 1], a0, a1, a2, a3, b2, b3);
      }
    }
    if (ch + 1 < nchunks) stage_v(ch + 1, cur ^ 1);
    cp_async_wait_all();
    __syncthreads();
  }
  // hi + lo, then the partial of this split: rows c0+cw+g (+8), columns j
#pragma unroll
  for (int nt = 0; nt < RPT; ++nt) {
    const int j = nt * 8 + 2 * q;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int c = c0 + cw + g + 8 * h;
      if (c < C) {
        float *dst = part + ((int64_t)blockIdx.y * C + c) * RPAD + j;
        dst[0] = d[nt][2 * h] + d[RPT + nt][2 * h];
        dst[1] = d[nt][2 * h + 1] + d[RPT + nt][2 * h + 1];
      }
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
  const int coltiles = (C + kGradCols - 1) / kGradCols;
  int64_t sp = (296 + coltiles - 1) / coltiles;
  int64_t maxsp = (M + kGradRows - 1) / kGradRows;
  if (sp > maxsp) sp = maxsp;
  if (sp < 1) sp = 1;
  return (int)sp;
}

template <int RPT>
static cudaError_t launch_grad(dim3 grid, const uint16_t *G, int64_t M, int C, const float *V,
                               int r, int64_t rps, float *part, cudaStream_t s) {
  const int smem = grad_smem_bytes(RPT * 8);
  static bool set = false;
  if (!set) {
    cudaError_t e = cudaFuncSetAttribute(lora_grad_tc_kernel<RPT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    set = true;
  }
  lora_grad_tc_kernel<RPT><<<grid, kGradThreads, smem, s>>>(G, M, C, V, r, rps, part);
  return cudaGetLastError();
}

cudaError_t launch_skinny(const uint16_t *G, int64_t M, int C, const float *V, int r, int RP,
                          float *part, int splits, cudaStream_t s) {
  const int64_t rps = ((M + splits - 1) / splits + kGradRows - 1) / kGradRows * kGradRows;
  dim3 grid((C + kGradCols - 1) / kGradCols, splits);
  switch (RP) {
    case 16: return launch_grad<2>(grid, G, M, C, V, r, rps, part, s);
    case 32: return launch_grad<4>(grid, G, M, C, V, r, rps, part, s);
    case 48: return launch_grad<6>(grid, G, M, C, V, r, rps, part, s);
    case 64: return launch_grad<8>(grid, G, M, C, V, r, rps, part, s);
    default: return cudaErrorInvalidValue;
  }
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
