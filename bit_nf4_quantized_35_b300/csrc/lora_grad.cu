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
// dst = s . G^T V  (transpose = 0: dst[c * r + j], the dB layout [N, r];
//                   transpose = 1: dst[j * C + c], the dA layout [r, K])
// One CTA = 128 columns c x one M split, 8 warps of 16 columns each.  The M
// range streams in 64-row chunks through a 4-deep cp.async ring holding the
// G tile [64 m][128 c] (rows padded to 272 B so ldmatrix rows hit distinct
// banks) and the raw fp32 V rows [64 m][r_pad]; before its MMAs a chunk's V
// is split into bf16 hi and lo rows of V^T [2 r_pad][64 m] (padded to
// 144 B).  The MMA A operand (16 c x 16 m) is an ldmatrix.trans of the G
// tile, the B operand (16 m x 8 j) an ldmatrix of V^T.
// Each split stores its fp32 partial sums part[split][c][j]; the last CTA of
// a column tile to finish (a counter per tile, left at zero) adds the splits
// in split order and writes dst, so the result does not depend on timing.
constexpr int kGradThreads = 256;
constexpr int kGradCols = 128;  // c per CTA
constexpr int kGradRows = 64;   // m per chunk
constexpr int kGradStages = 4;  // cp.async ring depth
constexpr int kGsPitch = 136;   // halves per G-tile row (128 + 8)
constexpr int kVtPitch = 72;    // halves per V^T row (64 + 8)

// A plain register function (no volatile): the compiler may interleave the
// MMAs with the fragment loads.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
  asm(
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

__host__ __device__ inline int grad_smem_bytes(int RPAD) {
  return kGradStages * (kGradRows * kGsPitch * 2 + kGradRows * RPAD * 4) +
         (2 * RPAD) * kVtPitch * 2 + 16;
}

// One launch may run two independent contractions (dB and dA of one
// backward): CTAs [0, tiles0 * splits0) take job 0, the rest job 1; a CTA's
// column tile and M split come from its index within its job.
template <int RPT>  // r_pad / 8
__global__ void __launch_bounds__(kGradThreads) lora_grad_tc_kernel(const SkinnyJob j0,
                                                                    const SkinnyJob j1,
                                                                    int64_t M, int r) {
  pdl_wait_release();
  const int n0 = j0.tiles * j0.splits;
  const bool second = (int)blockIdx.x >= n0;
  const SkinnyJob &jb = second ? j1 : j0;
  const int local = second ? (int)blockIdx.x - n0 : (int)blockIdx.x;
  const int tile = local % jb.tiles, split = local / jb.tiles, nsplits = jb.splits;
  const uint16_t *__restrict__ G = jb.G;
  const int C = jb.C;
  const float *__restrict__ V = jb.V;
  const int64_t rows_per_split = jb.rows_per_split;
  float *__restrict__ part = jb.part;
  int *__restrict__ tile_count = jb.tile_count;
  const float sc = jb.sc;
  const int transpose = jb.transpose;
  float *__restrict__ dst = jb.dst;
  const uint32_t *__restrict__ mask = jb.mask;
  const int wpr = jb.wpr;
  constexpr int RPAD = RPT * 8;
  constexpr int NJ = 2 * RPAD;  // hi rows then lo rows
  constexpr int NTT = NJ / 8;   // n8 tiles
  extern __shared__ __align__(16) uint8_t grad_smem[];
  uint16_t *gs = reinterpret_cast<uint16_t *>(grad_smem);  // [S][64][136]
  float *vraw = reinterpret_cast<float *>(gs + kGradStages * kGradRows * kGsPitch);  // [S][64][RPAD]
  uint16_t *vt = reinterpret_cast<uint16_t *>(vraw + kGradStages * kGradRows * RPAD);  // [NJ][72]
  int *last_flag = reinterpret_cast<int *>(vt + NJ * kVtPitch);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;
  const int c0 = tile * kGradCols;
  const int64_t m_lo = (int64_t)split * rows_per_split;
  const int64_t m_hi = min(M, m_lo + rows_per_split);
  const int nchunks = m_hi > m_lo ? (int)((m_hi - m_lo + kGradRows - 1) / kGradRows) : 0;

  // One chunk: 64 x 128 bf16 of G (1024 16-byte pieces) and 64 x r fp32 of
  // V (r / 4 pieces per row, r % 8 == 0); rows past the split read nothing
  // and land as zeros.  One commit group per call, empty past the end.
  auto issue = [&](int ch) {
    if (ch < nchunks) {
      const int buf = ch % kGradStages;
      const int64_t mb = m_lo + (int64_t)ch * kGradRows;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = threadIdx.x + u * kGradThreads;
        const int row = i >> 4, cc = (i & 15) * 8;
        const int64_t m = mb + row;
        const int c = c0 + cc;
        const bool ok = m < m_hi && c < C;
        cp_async16(smem_u32(gs + (buf * kGradRows + row) * kGsPitch + cc),
                   G + (ok ? m * C + c : 0), ok ? 16u : 0u);
      }
      for (int i = threadIdx.x; i < kGradRows * (RPAD / 4); i += kGradThreads) {
        const int row = i / (RPAD / 4), j4 = (i % (RPAD / 4)) * 4;
        const int64_t m = mb + row;
        const bool ok = m < m_hi && j4 < r;
        cp_async16(smem_u32(vraw + (buf * kGradRows + row) * RPAD + j4),
                   V + (ok ? m * r + j4 : 0), ok ? 16u : 0u);
      }
    }
    cp_async_commit();
  };

  float d[NTT][4];
#pragma unroll
  for (int nt = 0; nt < NTT; ++nt) d[nt][0] = d[nt][1] = d[nt][2] = d[nt][3] = 0.f;
#pragma unroll
  for (int ch = 0; ch < kGradStages - 1; ++ch) issue(ch);
  const int cw = warp * 16;  // this warp's 16 columns inside the tile
  // ldmatrix lane roles: matrix mi = lane >> 3, row within it lane & 7
  const int mi = lane >> 3, lr = lane & 7;
  // dropout: the keep words of a chunk's pieces (a piece of 8 columns is one
  // byte of a keep word), loaded one chunk ahead so that their latency is
  // hidden behind the previous chunk's MMAs
  uint32_t kwc[4], kwn[4];
  auto load_kw = [&](int chx, uint32_t (&kw)[4]) {
    const int64_t mb = m_lo + (int64_t)chx * kGradRows;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = threadIdx.x + u * kGradThreads;
      const int row = i >> 4, cc = (i & 15) * 8;
      const int64_t m = mb + row;
      const int c = c0 + cc;
      kw[u] = (m < m_hi && c < C) ? __ldg(mask + m * wpr + (c >> 5)) : 0xffffffffu;
    }
  };
  if (mask) load_kw(0, kwc);
  for (int ch = 0; ch < nchunks; ++ch) {
    const int cur = ch % kGradStages;
    cp_async_wait<kGradStages - 2>();  // this thread's copies of chunk ch have landed
    __syncthreads();                   // everyone's; chunk ch - 1 is fully consumed
    issue(ch + kGradStages - 1);       // into the buffer chunk ch - 1 used
    if (mask) {
      if (ch + 1 < nchunks) load_kw(ch + 1, kwn);
      // zero the dropped elements of G in chunk ch
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = threadIdx.x + u * kGradThreads;
        const int row = i >> 4, cc = (i & 15) * 8;
        const int c = c0 + cc;
        uint32_t mk[4];
        keep_masks((kwc[u] >> (c & 31)) & 0xffu, mk);
        const uint32_t a = smem_u32(gs + (cur * kGradRows + row) * kGsPitch + cc);
        const uint4 v = lds_v4(a);
        sts_v4(a, v.x & mk[0], v.y & mk[1], v.z & mk[2], v.w & mk[3]);
      }
      if (ch + 1 < nchunks)
#pragma unroll
        for (int u = 0; u < 4; ++u) kwc[u] = kwn[u];
    }
    // V rows of chunk ch -> bf16 hi / lo, transposed
    for (int i = threadIdx.x; i < kGradRows * RPAD; i += kGradThreads) {
      const int row = i / RPAD, j = i % RPAD;
      const float v = vraw[(cur * kGradRows + row) * RPAD + j];
      const __nv_bfloat16 hi = __float2bfloat16_rn(v);
      const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
      vt[j * kVtPitch + row] = __bfloat16_as_ushort(hi);
      vt[(RPAD + j) * kVtPitch + row] = __bfloat16_as_ushort(lo);
    }
    __syncthreads();
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
        ldsm_x4(smem_u32(vt + row * kVtPitch + col), b0, b1, b2, b3);
        mma_bf16_16816(d[2 * np], a0, a1, a2, a3, b0, b1);
        mma_bf16_16816(d[2 * np + 1], a0, a1, a2, a3, b2, b3);
      }
    }
  }
  cp_async_wait<0>();
  // hi + lo, then the partial of this split: rows c0+cw+g (+8), columns j
#pragma unroll
  for (int nt = 0; nt < RPT; ++nt) {
    const int j = nt * 8 + 2 * q;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int c = c0 + cw + g + 8 * h;
      if (c < C) {
        float *p = part + ((int64_t)split * C + c) * RPAD + j;
        __stcg(p, d[nt][2 * h] + d[RPT + nt][2 * h]);
        __stcg(p + 1, d[nt][2 * h + 1] + d[RPT + nt][2 * h + 1]);
      }
    }
  }
  // Count this split in; the last one for the tile adds the splits in order.
  // The block barrier orders every thread's partial stores before thread
  // 0's fence and count (one release per CTA); the reading threads are
  // ordered after thread 0's count by the next barrier.
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const int prev = atomicAdd(tile_count + tile, 1);
    const bool last = prev == nsplits - 1;
    if (last) atomicExch(tile_count + tile, 0);
    __threadfence();
    *last_flag = last ? 1 : 0;
  }
  __syncthreads();
  if (*last_flag == 0) return;
  // 4 consecutive j per thread (r % 8 == 0), 8 split loads in flight; the
  // sum runs in split order.
  const int ncols = min(kGradCols, C - c0);
  const int r4 = r / 4;
  const float4 *pbase = reinterpret_cast<const float4 *>(part);
  const int64_t sp_stride = (int64_t)C * (RPAD / 4);  // float4s per split
  for (int i = threadIdx.x; i < ncols * r4; i += kGradThreads) {
    // transposed (dA) output: consecutive threads along c, coalesced rows
    const int c = transpose ? c0 + i % ncols : c0 + i / r4;
    const int j4 = transpose ? (i / ncols) * 4 : (i % r4) * 4;
    const float4 *src = pbase + (int64_t)c * (RPAD / 4) + j4 / 4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    int sp = 0;
    for (; sp + 8 <= nsplits; sp += 8) {
      float4 w[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) w[k] = __ldcg(src + (int64_t)(sp + k) * sp_stride);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        acc.x += w[k].x;
        acc.y += w[k].y;
        acc.z += w[k].z;
        acc.w += w[k].w;
      }
    }
    for (; sp < nsplits; ++sp) {
      const float4 w = __ldcg(src + (int64_t)sp * sp_stride);
      acc.x += w.x;
      acc.y += w.y;
      acc.z += w.z;
      acc.w += w.w;
    }
    if (transpose) {
      dst[(int64_t)(j4 + 0) * C + c] = sc * acc.x;
      dst[(int64_t)(j4 + 1) * C + c] = sc * acc.y;
      dst[(int64_t)(j4 + 2) * C + c] = sc * acc.z;
      dst[(int64_t)(j4 + 3) * C + c] = sc * acc.w;
    } else {
      *reinterpret_cast<float4 *>(dst + (int64_t)c * r + j4) =
          make_float4(sc * acc.x, sc * acc.y, sc * acc.z, sc * acc.w);
    }
  }
}

// Both transposes of the LoRA factors in one launch (blocks [0, nb) do B,
// the rest A):
//   Bt[j][n] = B[n][j] and At[k][j] = A[j][k] for j < r; 0 for r <= j < RP.
__global__ void transpose_ab_kernel(const uint16_t *__restrict__ A, const uint16_t *__restrict__ B,
                                    int N, int K, int r, int RP, int nb, uint16_t *__restrict__ At,
                                    uint16_t *__restrict__ Bt) {
  pdl_wait_release();
  const bool doB = (int)blockIdx.x < nb;
  const int64_t total = doB ? (int64_t)RP * N : (int64_t)K * RP;
  const int64_t b0 = doB ? blockIdx.x : blockIdx.x - nb;
  const int64_t nblk = doB ? nb : gridDim.x - nb;
  for (int64_t i = b0 * blockDim.x + threadIdx.x; i < total; i += nblk * blockDim.x) {
    if (doB) {
      const int j = (int)(i / N), n = (int)(i % N);
      Bt[i] = j < r ? B[(int64_t)n * r + j] : (uint16_t)0;
    } else {
      const int k = (int)(i / RP), j = (int)(i % RP);
      At[i] = j < r ? A[(int64_t)j * K + k] : (uint16_t)0;
    }
  }
}

// ---------------------------------------------------------------------------
// LoRA down-projection out = G . H^T for a tall, skinny product:
//   forward  t = x . A^T   (G = x [M, K],  H = A  [r, K])
//   backward u = dY . B    (G = dY [M, N], H = B^T [r, N])
// It also writes bf16(s . out), zero-padded to r_pad columns: the operand of
// the rank-r MMAs that seed the fused GEMM's accumulator.
// One CTA per 16 rows of G (C < 8192), or a cluster of 2 CTAs per 16 rows,
// each CTA one half of C; a CTA's columns are split among its 16 warps;
// bf16 mma.sync m16n8k16 with fp32 accumulation (G streams from memory once,
// H is a few KB and stays in L1/L2).  The kernel is bound by HBM: each lane issues the loads
// of U 32-column chunks before the first MMA that needs them, so
// 16 warps x 32 lanes x 2U x 16 B of G are in flight per CTA.  The warp
// partials meet in shared memory in a fixed order (w + 8 first, then the
// 8 sums in warp order), then the two CTAs' sums in CTA 0 through
// distributed shared memory (CTA 0's half first).
// Lane (g, q) loads 8 consecutive elements (16 B) of rows g and g+8 per 32
// columns; the two MMAs of those 32 columns pair their k indices in the same
// order for G and H, so any consistent assignment is exact.
constexpr int kDownWarps = 16;

template <int NT>  // n8 tiles: r_pad / 8
__global__ void __launch_bounds__(kDownWarps * 32) lora_down_kernel(
    const uint16_t *__restrict__ G, int64_t M, int C, const uint16_t *__restrict__ H, int r,
    float s, float *__restrict__ out, uint16_t *__restrict__ outb, int r_pad,
    const uint32_t *__restrict__ mask, int wpr, float keep_scale) {
  pdl_wait_release();
  constexpr int U = NT <= 2 ? 4 : (NT <= 4 ? 2 : 1);  // chunks in flight per lane
  __shared__ float red[kDownWarps / 2][16][NT * 8];
  __shared__ float fin[16][NT * 8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;
  const int64_t m0 = (int64_t)blockIdx.x * 16;
  const int64_t rg = m0 + g, rg8 = m0 + g + 8;
  const bool vg = rg < M, vg8 = rg8 < M;
  // this CTA's part of C (all of it, or half: blockIdx.y = rank in the
  // cluster), then this warp's share of it, in 32-column chunks
  const int nch = (C + 31) / 32;
  const int h0 = gridDim.y == 2 ? (nch + 1) / 2 : nch;
  const int ch_lo = blockIdx.y == 0 ? 0 : h0, ch_n = blockIdx.y == 0 ? h0 : nch - h0;
  const int per = (ch_n + kDownWarps - 1) / kDownWarps;
  const int c_lo = (ch_lo + min(ch_n, warp * per)) * 32;
  const int c_hi = min(C, (ch_lo + min(ch_n, (warp + 1) * per)) * 32);
  float d[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) d[nt][0] = d[nt][1] = d[nt][2] = d[nt][3] = 0.f;
  const uint16_t *g0p = G + (vg ? rg : 0) * C;
  const uint16_t *g8p = G + (vg8 ? rg8 : 0) * C;
  for (int c0 = c_lo; c0 < c_hi; c0 += 32 * U) {
    uint4 a[U], b[U], h[U][NT];
    uint32_t ma[U], mb[U];  // dropout keep words of rows rg, rg8 (all ones without dropout)
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int cc = c0 + u * 32 + q * 8;
      const bool cv = cc < c_hi;  // C % 8 == 0
      a[u] = ldg_nc_v4(g0p + (cv ? cc : 0));
      b[u] = ldg_nc_v4(g8p + (cv ? cc : 0));
      ma[u] = mb[u] = 0xffffffffu;
      if (mask) {
        const int wd = (cv ? cc : 0) >> 5;
        ma[u] = __ldg(mask + (vg ? rg : 0) * wpr + wd);
        mb[u] = __ldg(mask + (vg8 ? rg8 : 0) * wpr + wd);
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int j = nt * 8 + g;
        h[u][nt] = ldg_nc_v4(H + (int64_t)(j < r ? j : 0) * C + (cv ? cc : 0));
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const bool cv = c0 + u * 32 + q * 8 < c_hi;
      const bool k0 = vg && cv, k8 = vg8 && cv;
      uint32_t A0[4] = {k0 ? a[u].x : 0u, k0 ? a[u].y : 0u, k0 ? a[u].z : 0u,
                        k0 ? a[u].w : 0u};
      uint32_t A8[4] = {k8 ? b[u].x : 0u, k8 ? b[u].y : 0u, k8 ? b[u].z : 0u,
                        k8 ? b[u].w : 0u};
      if (mask) {  // dropout: zero the dropped elements (byte q of the keep word)
        uint32_t m0[4], m8[4];
        keep_masks((ma[u] >> (8 * q)) & 0xffu, m0);
        keep_masks((mb[u] >> (8 * q)) & 0xffu, m8);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          A0[e] &= m0[e];
          A8[e] &= m8[e];
        }
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const bool hv = nt * 8 + g < r && cv;
        const uint4 hh = hv ? h[u][nt] : make_uint4(0, 0, 0, 0);
        // MMA 0: physical columns cc+0..3, MMA 1: cc+4..7
        mma_bf16_16816(d[nt], A0[0], A8[0], A0[1], A8[1], hh.x, hh.y);
        mma_bf16_16816(d[nt], A0[2], A8[2], A0[3], A8[3], hh.z, hh.w);
      }
    }
  }
  // Warps 8..15 store, warps 0..7 add theirs, then the 8 sums in warp order.
  const int wslot = warp & (kDownWarps / 2 - 1);
  for (int pass = 0; pass < 2; ++pass) {
    if ((warp >= kDownWarps / 2) == (pass == 0)) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        float *r0 = &red[wslot][g][nt * 8 + 2 * q];
        float *r8 = &red[wslot][g + 8][nt * 8 + 2 * q];
        if (pass == 0) {
          r0[0] = d[nt][0];
          r0[1] = d[nt][1];
          r8[0] = d[nt][2];
          r8[1] = d[nt][3];
        } else {
          r0[0] = d[nt][0] + r0[0];
          r0[1] = d[nt][1] + r0[1];
          r8[0] = d[nt][2] + r8[0];
          r8[1] = d[nt][3] + r8[1];
        }
      }
    }
    __syncthreads();
  }
  for (int i = threadIdx.x; i < 16 * NT * 8; i += blockDim.x) {
    const int row = i / (NT * 8), j = i % (NT * 8);
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kDownWarps / 2; ++w) v += red[w][row][j];
    fin[row][j] = v;
  }
  if (gridDim.y == 2) cluster_sync();  // both halves' sums are in shared memory
  if (blockIdx.y == 0) {
    for (int i = threadIdx.x; i < 16 * NT * 8; i += blockDim.x) {
      const int row = i / (NT * 8), j = i % (NT * 8);
      const int64_t m = m0 + row;
      if (m >= M) continue;
      float peer = 0.f;
      if (gridDim.y == 2)
        asm volatile("ld.shared::cluster.f32 %0, [%1];"
                     : "=f"(peer)
                     : "r"(mapa_shared(smem_u32(&fin[row][j]), 1))
                     : "memory");
      const float v = (fin[row][j] + peer) * keep_scale;
      if (out && j < r) out[m * r + j] = v;
      if (outb && j < r_pad)
        outb[m * r_pad + j] = j < r ? __bfloat16_as_ushort(__float2bfloat16_rn(s * v)) : (uint16_t)0;
    }
  }
  if (gridDim.y == 2) cluster_sync();  // the peer's sums are read before it exits
}

// ------------------------------------------------------------ launchers
template <int NT>
static cudaError_t launch_down(unsigned gx, const uint16_t *G, int64_t M, int C,
                               const uint16_t *H, int r, float s, float *out, uint16_t *outb,
                               int r_pad, const uint32_t *mask, int wpr, float keep_scale,
                               cudaStream_t st) {
  // Wide inputs: two CTAs per row block (a cluster), so that more SMs stream.
  const bool split = C >= 8192;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(gx, split ? 2 : 1, 1);
  cfg.blockDim = dim3(kDownWarps * 32, 1, 1);
  cfg.stream = st;
  cudaLaunchAttribute attrs[2];
  attrs[0] = pdl_attr();
  attrs[1].id = cudaLaunchAttributeClusterDimension;
  attrs[1].val.clusterDim.x = 1;
  attrs[1].val.clusterDim.y = 2;
  attrs[1].val.clusterDim.z = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = split ? 2 : 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, lora_down_kernel<NT>, G, M, C, H, r, s, out, outb,
                                     r_pad, mask, wpr, keep_scale);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_lora_down(const uint16_t *G, int64_t M, int C, const uint16_t *H, int r,
                             float s, float *out, uint16_t *outb, int r_pad, int num_sms,
                             cudaStream_t st, const uint32_t *mask, int wpr, float keep_scale) {
  (void)num_sms;
  if (M == 0) return cudaSuccess;
  const unsigned gx = (unsigned)((M + 15) / 16);
  const float ks = mask ? keep_scale : 1.0f;
  switch ((r + 7) / 8) {
    case 1:
    case 2: return launch_down<2>(gx, G, M, C, H, r, s, out, outb, r_pad, mask, wpr, ks, st);
    case 3:
    case 4: return launch_down<4>(gx, G, M, C, H, r, s, out, outb, r_pad, mask, wpr, ks, st);
    case 5:
    case 6: return launch_down<6>(gx, G, M, C, H, r, s, out, outb, r_pad, mask, wpr, ks, st);
    case 7:
    case 8: return launch_down<8>(gx, G, M, C, H, r, s, out, outb, r_pad, mask, wpr, ks, st);
    default: return cudaErrorInvalidValue;
  }
}

// ---------------------------------------------------------------------------
// The same down-projection for wide inputs (C >= 8192: the backward u = dY . B
// of the gate and up projections, the forward t of the down projection),
// where it runs about 25% faster than the register-streaming kernel above
// (which stays faster for narrower inputs, whose few stages per CTA leave
// the ring's fixed latency exposed).
// HBM-bound on G.  A CTA takes 16 rows of G and one of S column slices (a
// cluster of S CTAs per 16 rows, S chosen so that all CTAs are resident at
// once).  One producer lane streams its slice in 256-column stages through a
// ring in shared memory: TMA tensor loads in the 128-byte swizzle, four
// 64-column boxes of G (16 rows) and four of H (r_pad rows, zero past r) per
// stage, completion on the stage's mbarrier.  Four consumer warps take the
// stages in turn (warp w: stages w, w + 4, ..., always the same ring slots)
// and run bf16 mma.sync m16n8k16 on ldmatrix fragments with fp32
// accumulation; with LoRA dropout
// they zero the dropped elements of each G fragment first.  The warp partials
// are added in warp order, then the S slices in CTA 0 of the cluster in rank
// order through distributed shared memory, so the result does not depend on
// timing.  Every wait is bounded.
constexpr int kDownConsumers = 4;
constexpr int kDownThreads = (kDownConsumers + 1) * 32;
constexpr int kDownCols = 256;  // columns of G per stage

__host__ __device__ constexpr int down_stage_bytes(int NT) {
  return 4 * 16 * 128 + 4 * NT * 8 * 128;  // four G boxes, four H boxes
}
// Ring depth: a multiple of the consumer warps, so that every slot is only
// ever read by one warp (stage i -> slot i % depth, warp i % 4).  That warp
// then waits on a slot's full barrier only after it consumed the slot's
// previous phase, and the producer refills a slot only after that warp
// released it, so no wait can see a phase two ahead of the barrier (a 1-bit
// parity wait cannot tell those apart).
constexpr int kDownDepth = kDownConsumers;
static_assert(kDownDepth % kDownConsumers == 0, "one consumer warp per ring slot");
static int down_depth(int) { return kDownDepth; }
static int down_smem_bytes(int NT) {
  return 1024 + down_depth(NT) * down_stage_bytes(NT) + 2 * 8 * 8 + 16;
}

template <int NT>  // n8 tiles: r_pad / 8
__global__ void __launch_bounds__(kDownThreads) lora_down_tma_kernel(
    const __grid_constant__ CUtensorMap tmG, const __grid_constant__ CUtensorMap tmH, int64_t M,
    int C, int r, float s, float *__restrict__ out, uint16_t *__restrict__ outb, int r_pad,
    int S, int depth, int *status, const uint32_t *__restrict__ mask, int wpr,
    float keep_scale) {
  extern __shared__ uint8_t dsm_raw[];
  const uint32_t base = (smem_u32(dsm_raw) + 1023u) & ~1023u;
  float *ring = reinterpret_cast<float *>(dsm_raw + (base - smem_u32(dsm_raw)));
  constexpr int SB = down_stage_bytes(NT);
  constexpr int GB = 16 * 128;      // one G box: 64 columns x 16 rows
  constexpr int HB = NT * 8 * 128;  // one H box: 64 columns x r_pad rows
  const uint32_t bars = base + depth * SB;  // full[depth], then empty[depth]
  const uint32_t err = bars + 2 * depth * 8;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;
  const uint32_t rank = S > 1 ? cluster_rank() : 0u;
  const int64_t m0 = (int64_t)(blockIdx.x / S) * 16;
  const int nch = (C + kDownCols - 1) / kDownCols;
  const int k0 = (int)((int64_t)nch * rank / S), k1 = (int)((int64_t)nch * (rank + 1) / S);
  const int n = k1 - k0;  // stages of this CTA
  if (threadIdx.x < depth) {
    mbar_init(bars + threadIdx.x * 8, 1);
    mbar_init(bars + (depth + threadIdx.x) * 8, 1);
  }
  if (threadIdx.x == 0) st_shared_volatile(err, 0u);
  fence_barrier_init();
  __syncthreads();
  pdl_wait_release();

  float d[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) d[nt][0] = d[nt][1] = d[nt][2] = d[nt][3] = 0.f;
  if (warp == kDownConsumers) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmG);
      tma_prefetch_desc(&tmH);
      int i = 0;
      for (; i < n; ++i) {
        const int slot = i % depth;
        if (i >= depth &&
            !mbar_wait_bounded(bars + (depth + slot) * 8, (uint32_t)(i / depth - 1) & 1u, err,
                               status))
          break;
        const uint32_t st = base + slot * SB, full = bars + slot * 8;
        const int col = (k0 + i) * kDownCols;
        mbar_arrive_expect_tx(full, SB);
#pragma unroll
        for (int bx = 0; bx < 4; ++bx)
          tma_load_2d(st + bx * GB, &tmG, full, col + 64 * bx, (int)m0);
#pragma unroll
        for (int bx = 0; bx < 4; ++bx)
          tma_load_2d(st + 4 * GB + bx * HB, &tmH, full, col + 64 * bx, 0);
      }
      // error path: the copies still in flight land before the ring is reused
      if (ld_shared_volatile(err))
        for (int j = i > depth ? i - depth : 0; j < i; ++j)
          mbar_drain(bars + (j % depth) * 8, (uint32_t)(j / depth) & 1u);
    }
  } else {
    // ---------------------------------------------------- consumer warps
    const int64_t rg = m0 + g < M ? m0 + g : 0, rg8 = m0 + g + 8 < M ? m0 + g + 8 : 0;
    for (int i = warp; i < n; i += kDownConsumers) {
      const int slot = i % depth;
      const bool ok = __all_sync(
          0xffffffffu, mbar_wait_bounded(bars + slot * 8, (uint32_t)(i / depth) & 1u, err, status));
      if (!ok) break;
      const uint32_t st = base + slot * SB;
      const int col0 = (k0 + i) * kDownCols;
      uint32_t mw0 = 0xffffffffu, mw8 = 0xffffffffu;  // keep words of rows g, g + 8
#pragma unroll
      for (int ks = 0; ks < kDownCols / 16; ++ks) {
        const uint32_t gbox = st + (ks >> 2) * GB, hbox = st + 4 * GB + (ks >> 2) * HB;
        const int c0 = (ks & 3) * 2;  // first 16-byte chunk of the k step in a 128-byte row
        const int mi = lane >> 3, rr = lane & 7;
        uint32_t a0, a1, a2, a3;
        {
          const int row = rr + 8 * (mi & 1), ch = c0 + (mi >> 1);
          ldsm_x4(gbox + row * 128 + ((ch ^ (row & 7)) << 4), a0, a1, a2, a3);
        }
        if (mask) {  // dropout: zero the dropped elements of rows g, g + 8
          if ((ks & 1) == 0) {
            int wd = (col0 + ks * 16) >> 5;
            wd = wd < wpr ? wd : wpr - 1;  // columns past C hold zeros anyway
            mw0 = __ldg(mask + rg * wpr + wd);
            mw8 = __ldg(mask + rg8 * wpr + wd);
          }
          const int b = (ks & 1) * 16 + 2 * q;
          auto pm = [](uint32_t w, int sh) {
            const uint32_t k = (w >> sh) & 3u;
            return ((k & 1u) ? 0x0000ffffu : 0u) | ((k & 2u) ? 0xffff0000u : 0u);
          };
          a0 &= pm(mw0, b);
          a1 &= pm(mw8, b);
          a2 &= pm(mw0, b + 8);
          a3 &= pm(mw8, b + 8);
        }
#pragma unroll
        for (int np = 0; np < NT / 2; ++np) {
          const int row = (2 * np + (mi >> 1)) * 8 + rr, ch = c0 + (mi & 1);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(hbox + row * 128 + ((ch ^ (row & 7)) << 4), b0, b1, b2, b3);
          mma_bf16_16816(d[2 * np], a0, a1, a2, a3, b0, b1);
          mma_bf16_16816(d[2 * np + 1], a0, a1, a2, a3, b2, b3);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bars + (depth + slot) * 8);
    }
  }
  __syncthreads();  // every stage consumed: the ring is free for the sums
  constexpr int W = NT * 8;
  float *red = ring;                         // [consumer warp][16][W]
  float *fin = ring + kDownConsumers * 16 * W;  // [16][W]
  if (warp < kDownConsumers) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float *r0 = red + (warp * 16 + g) * W + nt * 8 + 2 * q;
      float *r8 = r0 + 8 * W;
      r0[0] = d[nt][0];
      r0[1] = d[nt][1];
      r8[0] = d[nt][2];
      r8[1] = d[nt][3];
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 16 * W; i += blockDim.x) {
    float v = red[i];
#pragma unroll
    for (int w = 1; w < kDownConsumers; ++w) v += red[w * 16 * W + i];
    fin[i] = v;
  }
  if (S > 1)
    cluster_sync();  // every slice's sums are in shared memory
  else
    __syncthreads();
  if (rank == 0) {
    for (int i = threadIdx.x; i < 16 * W; i += blockDim.x) {
      const int row = i / W, j = i - row * W;
      const int64_t m = m0 + row;
      if (m >= M) continue;
      float v = fin[i];
      for (int k = 1; k < S; ++k) {
        float peer;
        asm volatile("ld.shared::cluster.f32 %0, [%1];"
                     : "=f"(peer)
                     : "r"(mapa_shared(smem_u32(&fin[i]), (uint32_t)k))
                     : "memory");
        v += peer;
      }
      v *= keep_scale;
      if (out && j < r) out[m * r + j] = v;
      if (outb && j < r_pad)
        outb[m * r_pad + j] =
            j < r ? __bfloat16_as_ushort(__float2bfloat16_rn(s * v)) : (uint16_t)0;
    }
  }
  if (S > 1) cluster_sync();  // the peers' sums are read before they exit
}

template <int NT>
static cudaError_t launch_down_tma(const CUtensorMap &tmG, const CUtensorMap &tmH, int64_t M,
                                   int C, int r, float s, float *out, uint16_t *outb, int r_pad,
                                   int num_sms, int *status, const uint32_t *mask, int wpr,
                                   float keep_scale, cudaStream_t st) {
  const int depth = down_depth(NT), smem = down_smem_bytes(NT);
  static int occ = 0;  // resident CTAs per SM
  if (occ == 0) {
    cudaError_t e = cudaFuncSetAttribute(lora_down_tma_kernel<NT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    int o = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, lora_down_tma_kernel<NT>, kDownThreads,
                                                      smem);
    if (e != cudaSuccess) return e;
    occ = o > 0 ? o : 1;
  }
  // column slices per 16 rows: as many as keep every CTA resident at once,
  // at most 8 (a portable cluster) and at most one per stage
  const int64_t rt = (M + 15) / 16;
  const int nch = (C + kDownCols - 1) / kDownCols;
  int64_t S = (int64_t)num_sms * occ / rt;
  if (S > 8) S = 8;
  if (S > nch) S = nch;
  if (S < 1) S = 1;
  if (rt * S > 0x7fffffffLL) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(rt * S), 1, 1);
  cfg.blockDim = dim3(kDownThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attrs[2];
  attrs[0] = pdl_attr();
  attrs[1].id = cudaLaunchAttributeClusterDimension;
  attrs[1].val.clusterDim.x = (unsigned)S;
  attrs[1].val.clusterDim.y = 1;
  attrs[1].val.clusterDim.z = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = S > 1 ? 2 : 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, lora_down_tma_kernel<NT>, tmG, tmH, M, C, r, s, out,
                                     outb, r_pad, (int)S, depth, status, mask, wpr, keep_scale);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_lora_down_tma(const CUtensorMap &tmG, const CUtensorMap &tmH, int64_t M,
                                 int C, int r, float s, float *out, uint16_t *outb, int r_pad,
                                 int num_sms, int *status, cudaStream_t st, const uint32_t *mask,
                                 int wpr, float keep_scale) {
  if (M == 0) return cudaSuccess;
  const float ks = mask ? keep_scale : 1.0f;
  auto go = [&](auto launcher) {
    return launcher(tmG, tmH, M, C, r, s, out, outb, r_pad, num_sms, status, mask, wpr, ks, st);
  };
  switch ((r + 7) / 8) {
    case 1:
    case 2: return go(launch_down_tma<2>);
    case 3:
    case 4: return go(launch_down_tma<4>);
    case 5:
    case 6: return go(launch_down_tma<6>);
    case 7:
    case 8: return go(launch_down_tma<8>);
    default: return cudaErrorInvalidValue;
  }
}

// M splits per column tile: as many as keep all CTAs in one wave of two
// CTAs per SM (148 SMs), with at least 2 chunks of 64 rows per split.
int skinny_splits(int64_t M, int C, int budget) {
  const int coltiles = (C + kGradCols - 1) / kGradCols;
  int64_t sp = budget / (coltiles > 0 ? coltiles : 1);
  int64_t maxsp = (M + 2 * kGradRows - 1) / (2 * kGradRows);
  if (sp > maxsp) sp = maxsp;
  if (sp < 1) sp = 1;
  return (int)sp;
}

// dB (C = N) and dA (C = K) share one launch: the 296 CTAs of one wave (two
// per SM) are shared in proportion to their column tiles, so that every CTA
// gets about the same rows x columns.
void skinny_splits_pair(int64_t M, int N, int K, int *sn, int *sk) {
  const int tn = (N + kGradCols - 1) / kGradCols, tk = (K + kGradCols - 1) / kGradCols;
  const int tot = tn + tk > 0 ? tn + tk : 1;
  *sn = skinny_splits(M, N, 296 * tn / tot);
  *sk = skinny_splits(M, K, 296 * tk / tot);
}

int skinny_tiles(int C) { return (C + kGradCols - 1) / kGradCols; }

template <int RPT>
static cudaError_t launch_grad(const SkinnyJob &j0, const SkinnyJob &j1, int64_t M, int r,
                               cudaStream_t s) {
  const int smem = grad_smem_bytes(RPT * 8);
  static bool set = false;
  if (!set) {
    cudaError_t e = cudaFuncSetAttribute(lora_grad_tc_kernel<RPT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(j0.tiles * j0.splits + j1.tiles * j1.splits), 1, 1);
  cfg.blockDim = dim3(kGradThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attrs[1] = {pdl_attr()};
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, lora_grad_tc_kernel<RPT>, j0, j1, M, r);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

SkinnyJob skinny_job(const uint16_t *G, int64_t M, int C, const float *V, float *part,
                     int *tile_count, int splits, float sc, bool transpose, float *dst,
                     const uint32_t *mask, int wpr) {
  SkinnyJob j{};
  j.G = G;
  j.C = C;
  j.V = V;
  j.splits = C > 0 ? splits : 0;
  j.tiles = (C + kGradCols - 1) / kGradCols;
  j.rows_per_split = ((M + splits - 1) / splits + kGradRows - 1) / kGradRows * kGradRows;
  j.part = part;
  j.tile_count = tile_count;
  j.sc = sc;
  j.transpose = transpose ? 1 : 0;
  j.dst = dst;
  j.mask = mask;
  j.wpr = wpr;
  return j;
}

cudaError_t launch_skinny2(const SkinnyJob &j0, const SkinnyJob &j1, int64_t M, int r, int RP,
                           cudaStream_t s) {
  if (j0.tiles * j0.splits + j1.tiles * j1.splits == 0) return cudaSuccess;
  switch (RP) {
    case 16: return launch_grad<2>(j0, j1, M, r, s);
    case 32: return launch_grad<4>(j0, j1, M, r, s);
    case 48: return launch_grad<6>(j0, j1, M, r, s);
    case 64: return launch_grad<8>(j0, j1, M, r, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_skinny(const uint16_t *G, int64_t M, int C, const float *V, int r, int RP,
                          float *part, int *tile_count, int splits, float sc, bool transpose,
                          float *dst, cudaStream_t s, const uint32_t *mask, int wpr) {
  if (C == 0) return cudaSuccess;
  const SkinnyJob j0 = skinny_job(G, M, C, V, part, tile_count, splits, sc, transpose, dst, mask,
                                  wpr);
  SkinnyJob none{};
  none.tiles = 1;
  return launch_skinny2(j0, none, M, r, RP, s);
}

cudaError_t launch_transposes(const uint16_t *A, const uint16_t *B, int N, int K, int r, int RP,
                              uint16_t *At, uint16_t *Bt, int num_sms, cudaStream_t s) {
  const int64_t tb = (int64_t)RP * N, ta = (int64_t)K * RP;
  int64_t gb = (tb + 255) / 256, ga = (ta + 255) / 256;
  const int64_t cap = (int64_t)num_sms * 4;
  if (gb > cap) gb = cap;
  if (ga > cap) ga = cap;
  if (gb < 1) gb = 1;
  if (ga < 1) ga = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(gb + ga), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attrs[1] = {pdl_attr()};
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, transpose_ab_kernel, A, B, N, K, r, RP, (int)gb, At, Bt);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace qlora
