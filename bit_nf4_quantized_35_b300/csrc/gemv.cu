// gemv.cu -- memory-bound split-K QLoRA forward for decode-sized M (<= 16
// tokens), sm_103a.
//
// y[m, n] = sum_k x[m, k] w_hat[n, k] + s . sum_j t[m, j] B[n, j]
// ("QLoRA and 4bit Quantization | QLoRA 与 4-bit 量化", Step 3 formula).
//
// The packed 4-bit weight is the only large operand (N*K/2 bytes), so the
// kernel is built to stream it from HBM once at full width:
//   - A cluster of S CTAs (S <= 8) owns a contiguous range of 16-row tiles
//     of W; CTA s of the cluster and its warps each own one fixed 128-wide
//     slice of K, so a warp's x fragments are loaded into registers once.
//   - Per 64-weight block the block constant a_hat is factored out:
//       sum_{k in block} w_hat x = a_hat . sum_{k in block} c_idx(k) x_k,
//     and the inner sum runs on the tensor cores (mma.sync m16n8k16, f16
//     operands, f32 accumulation): the 4-bit indices become f16 codepoint
//     pairs through a 256-entry byte table in shared memory, replicated per
//     lane so that 32 random bytes never collide on a bank.
//   - x is converted to f16 with a per-token power-of-two scale chosen per
//     128-wide slice (exact; it keeps any bf16 magnitude in f16 range).
//   - The S partial sums of a tile meet in distributed shared memory: CTA 0
//     of the cluster adds them in rank order (deterministic), adds the LoRA
//     term from t (fp32) and B, and writes y.  No workspace, no atomics.
// The codepoints enter as f16 (error <= 2^-12 relative) and the product
// with a_hat stays in fp32, so the result is within the documented
// tolerance of x . W_hat^T with the bf16-rounded W_hat.
#include "common.cuh"
#include "kernels.h"

namespace qlora {

__constant__ float kNf4Const[16] = {QLORA_NF4_VALUES};

// Warps per CTA: 16 for up to 8 tokens; 12 for 9..16 tokens, whose larger
// register footprint needs the 168 registers a thread gets with 3 warps per
// SM sub-partition.
template <int NT>
struct GemvWarps {
  static constexpr int value = NT == 1 ? 16 : 12;
};


__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
__device__ __forceinline__ float ld_dsmem_f32(const float *local, uint32_t rank) {
  uint32_t la = smem_u32(local), ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(la), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
  return v;
}

// Codepoint pair of one packed byte: byte index 0..3 of word w, table
// address = byte * 128 + lane * 4.
template <int kByte>
__device__ __forceinline__ uint32_t lut(const uint8_t *tab, uint32_t w, uint32_t lane4) {
  uint32_t off;
  if constexpr (kByte == 0)
    off = ((w << 7) & 0x7f80u) | lane4;
  else
    off = ((w >> (8 * kByte - 7)) & 0x7f80u) | lane4;
  return *reinterpret_cast<const uint32_t *>(tab + off);
}

// bf16 pair -> f16 pair (both halves), round to nearest.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w, float sc = 1.0f) {
  return pack_f16x2(bf16_lo(w) * sc, bf16_hi(w) * sc);
}

// Shared-memory layout of the GEMV kernel (bytes).
struct GemvSmem {
  int tab, red, tpart, tfull, part, bsm, total;
};
__host__ __device__ inline GemvSmem gemv_smem_layout(int warps, int rows_max) {
  GemvSmem L;
  L.tab = 0;                                    // 256 x 32 lanes x u32
  L.red = 32768;                                // 2 x W x 32 rows x 16 tok f32 (also t staging)
  L.tpart = L.red + 2 * warps * 32 * 16 * 4;    // 64 j x 16 tok f32: this CTA's partial t
  L.tfull = L.tpart + 64 * 16 * 4;              // 16 tok x 64 j f32: full t (cluster rank 0)
  L.part = L.tfull + 16 * 64 * 4;               // rows_max x 16 tok f32: this CTA's partial y
  L.bsm = L.part + rows_max * 16 * 4;           // rows_max x 64 bf16: LoRA B rows (rank 0)
  L.total = L.bsm + rows_max * 64 * 2;
  return L;
}

template <int NT>
__global__ void __launch_bounds__(GemvWarps<NT>::value * 32, 1) qlora_gemv_kernel(const GemvArgs p) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int W = blockDim.x >> 5;
  const GemvSmem SL = gemv_smem_layout(W, p.rows_max);
  const uint8_t *tab = smem + SL.tab;
  float *red = reinterpret_cast<float *>(smem + SL.red);
  float *tpart = reinterpret_cast<float *>(smem + SL.tpart);
  float *tfull = reinterpret_cast<float *>(smem + SL.tfull);
  float *part = reinterpret_cast<float *>(smem + SL.part);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tq = lane & 3;
  const uint32_t rank = cluster_ctarank();
  const int S = gridDim.y;
  const int MT = NT * 8;
  const int RP = (p.r + 15) & ~15;

  // Codepoint-pair table: entry b holds f16(c[b >> 4]) (low half, element
  // 2j) and f16(c[b & 15]) (high half, element 2j+1), 32 copies.
  {
    uint32_t *t32 = reinterpret_cast<uint32_t *>(smem + SL.tab);
    for (int i = threadIdx.x; i < 256 * 32; i += blockDim.x) {
      const int b = i >> 5;
      t32[i] = pack_f16x2(kNf4Const[b >> 4], kNf4Const[b & 15]);
    }
  }

  const int rt_begin = (int)((int64_t)p.row_tiles * blockIdx.x / p.clusters);
  const int rt_end = (int)((int64_t)p.row_tiles * (blockIdx.x + 1) / p.clusters);
  const int row_lo = rt_begin * 16;
  const int row_hi = min(rt_end * 16, p.N);
  uint16_t *bsm = reinterpret_cast<uint16_t *>(smem + SL.bsm);
  if (rank == 0) {
    // LoRA B rows of this cluster's range, [row][j] with row stride 64
    const int nb = (row_hi - row_lo) * p.r;
    for (int i = threadIdx.x; i < nb; i += blockDim.x) {
      const int row = i / p.r, j = i % p.r;
      bsm[row * 64 + j] = p.B[(int64_t)(row_lo + row) * p.r + j];
    }
  }

  // This warp's 128-wide slice of K and its x fragments (f16, scaled by a
  // per-token power of two so any bf16 magnitude fits f16).
  const int chunk = (int)rank * W + warp;
  const int kc0 = chunk * 128;
  const bool kvalid = kc0 < p.K;
  uint32_t xf[2][4][NT][2];
  int xe[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int tok = nt * 8 + g;
    float v[2][16];
    float amax = 0.f;
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
      uint4 u0 = make_uint4(0, 0, 0, 0), u1 = u0;
      if (kc0 + blk * 64 < p.K && tok < p.M) {
        const uint16_t *src = p.x + (int64_t)tok * p.K + kc0 + blk * 64 + tq * 16;
        u0 = ldg_nc_v4(src);
        u1 = ldg_nc_v4(src + 8);
      }
      const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        v[blk][2 * e] = bf16_lo(w[e]);
        v[blk][2 * e + 1] = bf16_hi(w[e]);
        amax = fmaxf(amax, fmaxf(fabsf(v[blk][2 * e]), fabsf(v[blk][2 * e + 1])));
      }
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const int E = (int)((__float_as_uint(amax) >> 23) & 0xff) - 127;
    const int e = E >= 15 ? E - 14 : 0;
    xe[nt] = e;
    const float sc = __uint_as_float((uint32_t)(127 - e) << 23);  // 2^-e
#pragma unroll
    for (int blk = 0; blk < 2; ++blk)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        xf[blk][j][nt][0] = pack_f16x2(v[blk][4 * j] * sc, v[blk][4 * j + 1] * sc);
        xf[blk][j][nt][1] = pack_f16x2(v[blk][4 * j + 2] * sc, v[blk][4 * j + 3] * sc);
      }
  }
  // 2^e of the two tokens (nt*8 + 2tq, +1) whose accumulator columns this lane holds.
  float csc[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int e0 = __shfl_sync(0xffffffffu, xe[nt], (2 * tq) * 4);
    const int e1 = __shfl_sync(0xffffffffu, xe[nt], (2 * tq + 1) * 4);
    csc[nt][0] = __uint_as_float((uint32_t)(127 + e0) << 23);
    csc[nt][1] = __uint_as_float((uint32_t)(127 + e1) << 23);
  }

  // ---- LoRA down-projection t = x A^T on the tensor cores: rows j of A
  // play the weight rows, the same x fragments the tokens.
  for (int jt = 0; jt < RP / 16; ++jt) {
    float d[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) d[nt][0] = d[nt][1] = d[nt][2] = d[nt][3] = 0.f;
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
      uint32_t a0w[8], a8w[8];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int j = jt * 16 + g + 8 * h;
        uint4 u0 = make_uint4(0, 0, 0, 0), u1 = u0;
        if (j < p.r && kc0 + blk * 64 < p.K) {
          const uint16_t *src = p.A + (int64_t)j * p.K + kc0 + blk * 64 + tq * 16;
          u0 = ldg_nc_v4(src);
          u1 = ldg_nc_v4(src + 8);
        }
        uint32_t *dst = h ? a8w : a0w;
        dst[0] = u0.x, dst[1] = u0.y, dst[2] = u0.z, dst[3] = u0.w;
        dst[4] = u1.x, dst[5] = u1.y, dst[6] = u1.z, dst[7] = u1.w;
      }
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        // elements 4jj..4jj+3 of the lane's 16: words 2jj (k, k+1) and 2jj+1 (k+2, k+3)
        const uint32_t a[4] = {bf16x2_to_f16x2(a0w[2 * jj]), bf16x2_to_f16x2(a8w[2 * jj]),
                               bf16x2_to_f16x2(a0w[2 * jj + 1]), bf16x2_to_f16x2(a8w[2 * jj + 1])};
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_f16_16816(d[nt], a, xf[blk][jj][nt][0], xf[blk][jj][nt][1]);
      }
    }
    // stage this warp's partial t in `red` as [warp][j][tok]
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int tok = nt * 8 + 2 * tq;
      float *r0 = red + ((warp * 64) + jt * 16 + g) * 16 + tok;
      float *r8 = r0 + 8 * 16;
      r0[0] = d[nt][0] * csc[nt][0];
      r0[1] = d[nt][1] * csc[nt][1];
      r8[0] = d[nt][2] * csc[nt][0];
      r8[1] = d[nt][3] * csc[nt][1];
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < RP * 16; i += blockDim.x) {
    const int j = i >> 4, tok = i & 15;
    float v = 0.f;
    for (int w = 0; w < W; ++w) v += red[(w * 64 + j) * 16 + tok];
    tpart[i] = v;
  }
  cluster_sync_all();
  // Rank 0 of every cluster assembles the full t (fixed rank order); the
  // first cluster also saves it for the backward pass.
  if (rank == 0) {
    for (int i = threadIdx.x; i < 16 * RP; i += blockDim.x) {
      const int tok = i / RP, j = i % RP;
      float v = 0.f;
      for (int q = 0; q < S; ++q) v += ld_dsmem_f32(tpart + j * 16 + tok, (uint32_t)q);
      tfull[tok * 64 + j] = v;
      if (p.t_save && blockIdx.x == 0 && tok < p.M && j < p.r) p.t_save[tok * p.r + j] = v;
    }
  }
  __syncthreads();
  // Rank 0 seeds its partial y with the LoRA term s . t . B^T (fp32).
  if (rank == 0) {
    const int nrows = row_hi - row_lo;
    for (int i = threadIdx.x; i < nrows * MT; i += blockDim.x) {
      const int row = i / MT, tok = i % MT;
      float l = 0.f;
      for (int j = 0; j < p.r; ++j)
        l = fmaf(tfull[tok * 64 + j], __uint_as_float((uint32_t)bsm[row * 64 + j] << 16), l);
      part[row * 16 + tok] = p.s * l;
    }
  }

  // ---- main loop over pairs of 16-row tiles of this cluster's row range
  const uint32_t lane4 = lane * 4;
  const int64_t kblocks_row = p.K >> 6;
  const int n_it = (rt_end - rt_begin + 1) / 2;

  struct Piece {
    uint2 pk[2][2][2];  // [rt][row g / g+8][blk]
    int code[2][2][2];  // raw until use (see the GEMM producer)
    float cv[2][2][2];  // s2 (DQ) or fp32 absmax
    uint32_t valid;     // bit (rt*4 + h*2 + blk): block holds real weights
  };
  auto load_piece = [&](int it, Piece &P) {
    P.valid = 0;
#pragma unroll
    for (int rt = 0; rt < 2; ++rt)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int rtile = rt_begin + 2 * it + rt;
        const int row = rtile * 16 + g + 8 * h;
        const bool ok = it < n_it && rtile < rt_end && row < p.N && kvalid;
        // unconditional loads from a clamped address; validity applied at use
        const int rowc = ok ? row : 0;
#pragma unroll
        for (int blk = 0; blk < 2; ++blk) {
          const bool okb = ok && kc0 + blk * 64 < p.K;
          const int64_t kb = okb ? (kc0 >> 6) + blk : 0;
          P.pk[rt][h][blk] = ldg_nc_v2(p.packed + (int64_t)rowc * (p.K >> 1) + (kb << 5) + tq * 8);
          const int64_t b = (int64_t)rowc * kblocks_row + kb;
          P.code[rt][h][blk] = ldg_nc_s8(p.codes + (p.use_code ? b : 0));
          P.valid |= okb ? (1u << (rt * 4 + h * 2 + blk)) : 0u;
          P.cv[rt][h][blk] = ldg_nc_f32(p.cvec + (b >> p.cshift));
        }
      }
  };
  auto compute_piece = [&](int it, const Piece &P) {
    float acc[2][NT][4];
#pragma unroll
    for (int rt = 0; rt < 2; ++rt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[rt][nt][i] = 0.f;
#pragma unroll
    for (int rt = 0; rt < 2; ++rt)
#pragma unroll
      for (int blk = 0; blk < 2; ++blk) {
        float tmp[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) tmp[nt][0] = tmp[nt][1] = tmp[nt][2] = tmp[nt][3] = 0.f;
        const uint32_t w0[2] = {P.pk[rt][0][blk].x, P.pk[rt][0][blk].y};
        const uint32_t w8[2] = {P.pk[rt][1][blk].x, P.pk[rt][1][blk].y};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int wi = j >> 1;
          uint32_t a[4];
          if ((j & 1) == 0) {
            a[0] = lut<0>(tab, w0[wi], lane4);
            a[1] = lut<0>(tab, w8[wi], lane4);
            a[2] = lut<1>(tab, w0[wi], lane4);
            a[3] = lut<1>(tab, w8[wi], lane4);
          } else {
            a[0] = lut<2>(tab, w0[wi], lane4);
            a[1] = lut<2>(tab, w8[wi], lane4);
            a[2] = lut<3>(tab, w0[wi], lane4);
            a[3] = lut<3>(tab, w8[wi], lane4);
          }
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma_f16_16816(tmp[nt], a, xf[blk][j][nt][0], xf[blk][j][nt][1]);
        }
        const float ah0 = ((P.valid >> (rt * 4 + blk)) & 1u ? 1.0f : 0.0f) * (p.use_code ? __fmul_rn((float)P.code[rt][0][blk],
                                                                      P.cv[rt][0][blk])
                                                            : P.cv[rt][0][blk]);
        const float ah8 = ((P.valid >> (rt * 4 + 2 + blk)) & 1u ? 1.0f : 0.0f) * (p.use_code ? __fmul_rn((float)P.code[rt][1][blk],
                                                                      P.cv[rt][1][blk])
                                                            : P.cv[rt][1][blk]);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          acc[rt][nt][0] = fmaf(ah0, tmp[nt][0], acc[rt][nt][0]);
          acc[rt][nt][1] = fmaf(ah0, tmp[nt][1], acc[rt][nt][1]);
          acc[rt][nt][2] = fmaf(ah8, tmp[nt][2], acc[rt][nt][2]);
          acc[rt][nt][3] = fmaf(ah8, tmp[nt][3], acc[rt][nt][3]);
        }
      }
    float *rb = red + (it & 1) * (W * 32 * 16);
#pragma unroll
    for (int rt = 0; rt < 2; ++rt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int tok = nt * 8 + 2 * tq;
        float *r0 = rb + ((warp * 32) + rt * 16 + g) * 16 + tok;
        float *r8 = r0 + 8 * 16;
        *reinterpret_cast<float2 *>(r0) =
            make_float2(acc[rt][nt][0] * csc[nt][0], acc[rt][nt][1] * csc[nt][1]);
        *reinterpret_cast<float2 *>(r8) =
            make_float2(acc[rt][nt][2] * csc[nt][0], acc[rt][nt][3] * csc[nt][1]);
      }
    __syncthreads();
    // warp partials of these 32 rows -> this CTA's partial y (fixed order)
    const int rows_here = min(32, (rt_end - rt_begin - 2 * it) * 16);
    for (int i = threadIdx.x; i < rows_here * MT; i += blockDim.x) {
      const int row = i / MT, tok = i % MT;
      float v = 0.f;
      for (int w = 0; w < W; ++w) v += rb[(w * 32 + row) * 16 + tok];
      float *dst = part + (2 * it * 16 + row) * 16 + tok;
      *dst = (rank == 0) ? *dst + v : v;
    }
  };

  // Two-slot prefetch ring, compile-time slot indices.
  Piece P[2];
  load_piece(0, P[0]);
  for (int it0 = 0; it0 < n_it; it0 += 2) {
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int it = it0 + u;
      if (it < n_it) {
        load_piece(it + 1, P[(u + 1) & 1]);
        compute_piece(it, P[u]);
      }
    }
  }
  __syncthreads();
  cluster_sync_all();
  if (rank == 0) {
    const int nrows = row_hi - row_lo;
    for (int i = threadIdx.x; i < nrows * p.M; i += blockDim.x) {
      const int tok = i / nrows, row = i % nrows;
      float v = 0.f;
      for (int q = 0; q < S; ++q) v += ld_dsmem_f32(part + row * 16 + tok, (uint32_t)q);
      const int n = row_lo + row;
      if (p.y_bf16)
        reinterpret_cast<__nv_bfloat16 *>(p.y)[(int64_t)tok * p.N + n] = __float2bfloat16_rn(v);
      else
        reinterpret_cast<float *>(p.y)[(int64_t)tok * p.N + n] = v;
    }
  }
  cluster_sync_all();  // keep every CTA's shared memory alive until rank 0 has read it
}

// ------------------------------------------------------------ launchers
int gemv_plan(int K, int M, int *warps, int *S) {
  const int maxw = M > 8 ? GemvWarps<2>::value : GemvWarps<1>::value;
  const int chunks = (K + 127) / 128;
  int s = (chunks + maxw - 1) / maxw;
  if (s > 8) return -1;
  if (s < 1) s = 1;
  const int w = (chunks + s - 1) / s;
  *warps = w;
  *S = s;
  return 0;
}

cudaError_t launch_gemv(GemvArgs a, int num_sms, cudaStream_t s) {
  int warps, S;
  if (a.M < 1 || a.M > 16 || gemv_plan(a.K, a.M, &warps, &S) != 0) return cudaErrorInvalidValue;
  a.row_tiles = (a.N + 15) / 16;
  int clusters = num_sms / S;
  const int need = (a.row_tiles + 1) / 2;
  if (clusters > need) clusters = need;
  if (clusters < 1) clusters = 1;
  a.clusters = clusters;
  a.rows_max = ((a.row_tiles + clusters - 1) / clusters + 1) * 16;
  const size_t smem = gemv_smem_layout(warps, a.rows_max).total;
  if (smem > 232448) return cudaErrorInvalidValue;
  static bool attr[2] = {false, false};
  const int nt = a.M > 8 ? 2 : 1;
  cudaError_t e;
  if (!attr[nt - 1]) {
    if (nt == 2)
      e = cudaFuncSetAttribute(qlora_gemv_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               232448);
    else
      e = cudaFuncSetAttribute(qlora_gemv_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               232448);
    if (e != cudaSuccess) return e;
    if (nt == 2)
      e = cudaFuncSetAttribute(qlora_gemv_kernel<2>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    else
      e = cudaFuncSetAttribute(qlora_gemv_kernel<1>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    attr[nt - 1] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(clusters, S, 1);
  cfg.blockDim = dim3(warps * 32, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = 1;
  attrs[0].val.clusterDim.y = S;
  attrs[0].val.clusterDim.z = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  if (nt == 2)
    e = cudaLaunchKernelEx(&cfg, qlora_gemv_kernel<2>, a);
  else
    e = cudaLaunchKernelEx(&cfg, qlora_gemv_kernel<1>, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}


}  // namespace qlora
