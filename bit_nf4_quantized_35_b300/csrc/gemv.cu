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

constexpr int kGemvMaxWarps = 16;


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

template <int NT>
__global__ void __launch_bounds__(kGemvMaxWarps * 32, 1) qlora_gemv_kernel(const GemvArgs p) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint8_t *tab = smem;                                                   // 32 KB
  float *red = reinterpret_cast<float *>(smem + 32768);                 // [W][64][16]
  const int W = blockDim.x >> 5;
  float *part = red + W * 64 * 16;                                       // [64][16]
  float *t_s = part + 64 * 16;                                           // [16][r]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tq = lane & 3;
  const uint32_t rank = cluster_ctarank();
  const int S = gridDim.y;

  // Codepoint-pair table: entry b holds f16(c[b >> 4]) (low half, element
  // 2j) and f16(c[b & 15]) (high half, element 2j+1), 32 copies.
  {
    constexpr float c[16] = {QLORA_NF4_VALUES};
    for (int i = threadIdx.x; i < 256 * 32; i += blockDim.x) {
      const int b = i >> 5;
      float lo = 0.f, hi = 0.f;
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        if ((b >> 4) == q) lo = c[q];
        if ((b & 15) == q) hi = c[q];
      }
      reinterpret_cast<uint32_t *>(tab)[i] = pack_f16x2(lo, hi);
    }
    for (int i = threadIdx.x; i < p.M * p.r; i += blockDim.x) t_s[i] = p.t[i];
  }

  // This warp's 128-wide slice of K and its x fragments (f16, scaled).
  const int chunk = (int)rank * W + warp;
  const int kc0 = chunk * 128;
  const bool kvalid = kc0 < p.K;
  uint32_t xf[2][4][NT][2];
  int xe[NT];  // per-token exponent shift of this lane's token (nt*8 + g)
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
  // Scale factors 2^e of the two tokens (nt*8 + 2tq, +1) whose C columns this lane holds.
  float csc[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int e0 = __shfl_sync(0xffffffffu, xe[nt], (2 * tq) * 4);
    const int e1 = __shfl_sync(0xffffffffu, xe[nt], (2 * tq + 1) * 4);
    csc[nt][0] = __uint_as_float((uint32_t)(127 + e0) << 23);
    csc[nt][1] = __uint_as_float((uint32_t)(127 + e1) << 23);
  }
  __syncthreads();

  const uint32_t lane4 = lane * 4;
  const int64_t kblocks_row = p.K >> 6;
  const int MT = NT * 8;
  // Contiguous share of row tiles for this cluster.
  const int rt_begin = (int)((int64_t)p.row_tiles * blockIdx.x / p.clusters);
  const int rt_end = (int)((int64_t)p.row_tiles * (blockIdx.x + 1) / p.clusters);

  for (int rt0 = rt_begin; rt0 < rt_end; rt0 += 4) {
    // ---- loads: 4 row tiles x rows (g, g+8) x 2 blocks, 8 bytes each
    uint2 pk[4][2][2];
    float ah[4][2][2];
#pragma unroll
    for (int rt = 0; rt < 4; ++rt)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int row = (rt0 + rt) * 16 + g + 8 * h;
        const bool ok = kvalid && (rt0 + rt) < rt_end && row < p.N;
#pragma unroll
        for (int blk = 0; blk < 2; ++blk) {
          pk[rt][h][blk] = make_uint2(0, 0);
          ah[rt][h][blk] = 0.f;
          if (ok && kc0 + blk * 64 < p.K) {
            const int64_t kb = (kc0 >> 6) + blk;
            pk[rt][h][blk] =
                ldg_nc_v2(p.packed + (int64_t)row * (p.K >> 1) + (kb << 5) + tq * 8);
            const int64_t b = (int64_t)row * kblocks_row + kb;
            ah[rt][h][blk] = p.group > 0 ? __fmul_rn((float)__ldg(p.codes + b),
                                                     __ldg(p.scale2 + b / p.group))
                                         : __ldg(p.absf + b);
          }
        }
      }
    // ---- tensor-core partial sums
    float acc[4][NT][4];
#pragma unroll
    for (int rt = 0; rt < 4; ++rt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[rt][nt][i] = 0.f;
#pragma unroll
    for (int rt = 0; rt < 4; ++rt)
#pragma unroll
      for (int blk = 0; blk < 2; ++blk) {
        float tmp[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int i = 0; i < 4; ++i) tmp[nt][i] = 0.f;
        const uint32_t w0[2] = {pk[rt][0][blk].x, pk[rt][0][blk].y};
        const uint32_t w8[2] = {pk[rt][1][blk].x, pk[rt][1][blk].y};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          // bytes 2j and 2j+1 of the lane's 8-byte piece
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
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          acc[rt][nt][0] = fmaf(ah[rt][0][blk], tmp[nt][0], acc[rt][nt][0]);
          acc[rt][nt][1] = fmaf(ah[rt][0][blk], tmp[nt][1], acc[rt][nt][1]);
          acc[rt][nt][2] = fmaf(ah[rt][1][blk], tmp[nt][2], acc[rt][nt][2]);
          acc[rt][nt][3] = fmaf(ah[rt][1][blk], tmp[nt][3], acc[rt][nt][3]);
        }
      }
    // ---- warp partials -> shared memory
#pragma unroll
    for (int rt = 0; rt < 4; ++rt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int tok = nt * 8 + 2 * tq;
        float *r0 = red + ((warp * 64) + rt * 16 + g) * 16 + tok;
        float *r8 = r0 + 8 * 16;
        *reinterpret_cast<float2 *>(r0) =
            make_float2(acc[rt][nt][0] * csc[nt][0], acc[rt][nt][1] * csc[nt][1]);
        *reinterpret_cast<float2 *>(r8) =
            make_float2(acc[rt][nt][2] * csc[nt][0], acc[rt][nt][3] * csc[nt][1]);
      }
    __syncthreads();
    for (int i = threadIdx.x; i < 64 * MT; i += blockDim.x) {
      const int row = i / MT, tok = i % MT;
      float v = 0.f;
      for (int w = 0; w < W; ++w) v += red[(w * 64 + row) * 16 + tok];
      part[row * 16 + tok] = v;
    }
    cluster_sync_all();
    if (rank == 0) {
      const int row_lo = rt0 * 16;
      int row_hi = min(rt0 + 4, rt_end) * 16;
      if (row_hi > p.N) row_hi = p.N;
      const int nrows = row_hi - row_lo;
      for (int i = threadIdx.x; i < nrows * p.M; i += blockDim.x) {
        const int tok = i / nrows, row = i % nrows;
        float v = 0.f;
        for (int q = 0; q < S; ++q) v += ld_dsmem_f32(part + row * 16 + tok, (uint32_t)q);
        const int n = row_lo + row;
        float l = 0.f;
        const uint16_t *Bn = p.B + (int64_t)n * p.r;
        for (int jj = 0; jj < p.r; ++jj)
          l = fmaf(t_s[tok * p.r + jj], __uint_as_float((uint32_t)Bn[jj] << 16), l);
        v = v + p.s * l;
        if (p.y_bf16)
          reinterpret_cast<__nv_bfloat16 *>(p.y)[(int64_t)tok * p.N + n] = __float2bfloat16_rn(v);
        else
          reinterpret_cast<float *>(p.y)[(int64_t)tok * p.N + n] = v;
      }
    }
    cluster_sync_all();
  }
}

// t[m, j] = sum_k x[m, k] A[j, k]  (fp32 accumulation), one warp per (m, j).
__global__ void __launch_bounds__(256) lora_down_kernel(const uint16_t *__restrict__ x,
                                                        const uint16_t *__restrict__ A, int M,
                                                        int K, int r, float *__restrict__ t) {
  const int64_t wid = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= (int64_t)M * r) return;
  const int64_t m = wid / r;
  const int j = (int)(wid % r);
  const uint16_t *xr = x + m * K;
  const uint16_t *ar = A + (int64_t)j * K;
  float acc = 0.f;
  for (int k = lane * 8; k < K; k += 256) {
    const uint4 xv = ldg_nc_v4(xr + k), av = ldg_nc_v4(ar + k);
    const uint32_t xa[4] = {xv.x, xv.y, xv.z, xv.w}, aa[4] = {av.x, av.y, av.z, av.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      acc = fmaf(bf16_lo(xa[e]), bf16_lo(aa[e]), acc);
      acc = fmaf(bf16_hi(xa[e]), bf16_hi(aa[e]), acc);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) t[m * r + j] = acc;
}

// ------------------------------------------------------------ launchers
int gemv_plan(int K, int *warps, int *S) {
  const int chunks = (K + 127) / 128;
  int s = (chunks + kGemvMaxWarps - 1) / kGemvMaxWarps;
  if (s > 8) return -1;
  if (s < 1) s = 1;
  const int w = (chunks + s - 1) / s;
  *warps = w;
  *S = s;
  return 0;
}

size_t gemv_smem_bytes(int warps, int r) {
  return 32768 + (size_t)warps * 64 * 16 * 4 + 64 * 16 * 4 + (size_t)16 * r * 4;
}

cudaError_t launch_gemv(GemvArgs a, int num_sms, cudaStream_t s) {
  int warps, S;
  if (gemv_plan(a.K, &warps, &S) != 0) return cudaErrorInvalidValue;
  a.row_tiles = (a.N + 15) / 16;
  int clusters = num_sms / S;
  const int need = (a.row_tiles + 3) / 4;
  if (clusters > need) clusters = need;
  if (clusters < 1) clusters = 1;
  a.clusters = clusters;
  const size_t smem = gemv_smem_bytes(warps, a.r);
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

cudaError_t launch_lora_down(const uint16_t *x, const uint16_t *A, int64_t M, int K, int r,
                             float *t, cudaStream_t s) {
  const int64_t warps = M * r;
  if (warps == 0) return cudaSuccess;
  const int64_t blocks = (warps * 32 + 255) / 256;
  lora_down_kernel<<<(unsigned)blocks, 256, 0, s>>>(x, A, (int)M, K, r, t);
  return cudaGetLastError();
}

}  // namespace qlora
