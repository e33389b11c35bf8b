// gemm_tc.cu -- fused dequantise + tcgen05 GEMM + LoRA bypass for sm_103a.
//
// One kernel serves both dense contractions of the QLoRA linear layer
// ("QLoRA and 4bit Quantization | QLoRA 与 4-bit 量化", Step 3 formula and the
// gradient routing of Step 4's frozen-base test):
//   forward  (kDx = false): out[M, N] = x[M, K] . W_hat[N, K]^T
//                           aux[M, r] = x . A^T                 (t, saved)
//                           out     += (s . aux) . B^T          (LoRA, s = alpha/r)
//   backward (kDx = true) : out[M, K] = dY[M, N] . W_hat[N, K]
//                           aux[M, r] = dY . B                  (u, saved)
//                           out     += (s . aux) . A
//
// Tile 128 (M) x 256 (output columns), contraction step 64, one CTA per SM.
// Warp roles (320 threads):
//   warps 0-7  dequantising producers: every thread turns the 32 packed
//              bytes of one (row, 64-block) into 64 bf16 values through the
//              per-block table T[i] = bf16(c_i * a_hat) (byte permutes, no
//              smem lookups) and stores them straight into the B operand
//              tile in the 128-byte-swizzled layout the tensor core reads
//              (K-major for the forward, MN-major for dX).  After the main
//              loop the same warps run the epilogue.
//   warp 8     TMA producer: activation tile (x or dY) and the rank-r
//              down-projection tile per stage; the up-projection tile once.
//   warp 9     TMEM owner and single-thread tcgen05.mma issuer.
// Per stage the MMA thread issues 4 x (128x256x16) for the base product and
// 4 x (128 x r_pad x 16) for the LoRA down-projection, both reading the same
// activation tile, accumulating in TMEM columns [0,256) and [256,256+r_pad).
// After the contraction the epilogue warps read the down-projection, scale
// it by s, round it to bf16 into shared memory, and the MMA thread adds the
// rank-r up-projection into the base accumulator with r_pad/16 more MMAs
// before the final TMEM -> register -> global store.
//
// Every mbarrier wait is bounded (common.cuh): a wait that runs out writes
// QLORA_ERR_TIMEOUT to the device status word and every role runs to the
// end of the kernel without blocking, so the context stays usable.
#include "common.cuh"
#include "kernels.h"

namespace qlora {

constexpr int GBM = 128, GBN = 256, GBK = 64;
constexpr int kGemmThreads = 320;
constexpr int kABytes = GBM * GBK * 2;  // 16 KB
constexpr int kBBytes = GBN * GBK * 2;  // 32 KB

__host__ __device__ inline int gemm_stage_bytes(int r_pad) { return kABytes + kBBytes + r_pad * 128; }
__host__ __device__ inline int gemm_upa_bytes(int r_pad) { return (r_pad / 16) * GBM * 32; }
__host__ __device__ inline int gemm_upb_bytes(int r_pad) { return (r_pad / 16) * GBN * 32; }
__host__ inline int gemm_smem_bytes(int stages, int r_pad) {
  return 1024 + stages * gemm_stage_bytes(r_pad) + gemm_upa_bytes(r_pad) + gemm_upb_bytes(r_pad) +
         256;
}


// Raw packed bytes + block constant of one (row, 64-block) for one stage.
struct Fetch {
  uint4 lo, hi;
  float c;   // code (DQ) or fp32 absmax
  float s2;  // second-level scale (DQ) or 1
  bool valid;
};

__device__ __forceinline__ Fetch fetch_block(const GemmArgs &p, int64_t n, int64_t kcol,
                                             bool valid) {
  Fetch f;
  f.valid = valid;
  f.lo = make_uint4(0, 0, 0, 0);
  f.hi = f.lo;
  f.c = 0.0f;
  f.s2 = 1.0f;
  if (valid) {
    const uint8_t *src = p.packed + n * (p.wcols >> 1) + (kcol >> 1);
    f.lo = ldg_nc_v4(src);
    f.hi = ldg_nc_v4(src + 16);
    const int64_t blk = n * (p.wcols >> 6) + (kcol >> 6);
    if (p.group > 0) {
      f.c = (float)__ldg(p.codes + blk);
      f.s2 = __ldg(p.scale2 + blk / p.group);
    } else {
      f.c = __ldg(p.absf + blk);
    }
  }
  return f;
}

// Dequantise one fetched block into 64 bf16 values and store them as the
// 8 16-byte chunks of one 128-byte swizzled row at `row_addr` (chunk c goes
// to position c ^ swz).
__device__ __forceinline__ void dequant_store_row(const GemmArgs &p, const Fetch &f,
                                                  uint32_t row_addr, uint32_t swz) {
  if (!f.valid) {
#pragma unroll
    for (int c = 0; c < 8; ++c) sts_v4(row_addr + ((c ^ swz) << 4), 0, 0, 0, 0);
    return;
  }
  const float ahat = (p.group > 0) ? __fmul_rn(f.c, f.s2) : f.c;
  const Nf4Table t = make_table(ahat);
  const uint32_t w[8] = {f.lo.x, f.lo.y, f.lo.z, f.lo.w, f.hi.x, f.hi.y, f.hi.z, f.hi.w};
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    uint32_t o[4];
    lookup8(t, w[c], o);
    sts_v4(row_addr + ((c ^ swz) << 4), o[0], o[1], o[2], o[3]);
  }
}

// Bounded drain used only on the error path: waits for a phase regardless
// of the CTA error flag, for at most ~0.1 s.
__device__ __forceinline__ void mbar_drain(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > (1ll << 28)) return;
  }
}

template <bool kDx>
__global__ void __launch_bounds__(kGemmThreads, 1)
    qlora_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmL1,
                      const __grid_constant__ CUtensorMap tmL2, const GemmArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int S = p.stages, RP = p.r_pad;
  const int SB = gemm_stage_bytes(RP);
  uint8_t *upa = smem + S * SB;
  uint8_t *upb = upa + gemm_upa_bytes(RP);
  uint64_t *bars = reinterpret_cast<uint64_t *>(upb + gemm_upb_bytes(RP));
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * S + 4);
  volatile int *cta_err = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const uint32_t smem0 = smem_u32(smem);
  const uint32_t upa_u = smem_u32(upa), upb_u = smem_u32(upb);
  auto full_bar = [&](int s) { return smem_u32(bars + s); };
  auto empty_bar = [&](int s) { return smem_u32(bars + S + s); };
  const uint32_t upa_bar = smem_u32(bars + 2 * S), upb_bar = smem_u32(bars + 2 * S + 1);
  const uint32_t acc_bar = smem_u32(bars + 2 * S + 2), acc2_bar = smem_u32(bars + 2 * S + 3);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.y * GBM, c0 = blockIdx.x * GBN;
  const int num_k = (p.kdim + GBK - 1) / GBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1 + 8);  // TMA expect_tx arrive + 8 producer warps
      mbar_init(empty_bar(s), 1);     // tcgen05.commit
    }
    mbar_init(upa_bar, 4);
    mbar_init(upb_bar, 1);
    mbar_init(acc_bar, 1);
    mbar_init(acc2_bar, 1);
    *cta_err = 0;
    fence_barrier_init();
  }
  if (warp == 8 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmL1);
    tma_prefetch_desc(&tmL2);
  }
  if (warp == 9) tmem_alloc(smem_u32(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tmem_aux = tmem + 256;

  if (warp < 8) {
    // ------------------------------------------------ dequantising producers
    const int pid = threadIdx.x;  // 0..255
    int64_t n_fixed = 0, kcol_fixed = 0;
    uint32_t row_off, swz;
    int nl = 0;
    if (!kDx) {
      n_fixed = (int64_t)c0 + pid;  // weight row = output column
      row_off = (pid >> 3) * 1024 + (pid & 7) * 128;
      swz = pid & 7;
    } else {
      const int bsub = pid >> 6;  // which 64-column atom of the 256 outputs
      nl = pid & 63;              // contraction row inside the stage
      kcol_fixed = (int64_t)c0 + 64 * bsub;
      row_off = bsub * 8192 + (nl >> 3) * 1024 + (nl & 7) * 128;
      swz = nl & 7;
    }
    auto fetch_k = [&](int kb) -> Fetch {
      if (kb >= num_k) return fetch_block(p, 0, 0, false);
      if (!kDx) {
        const int64_t kcol = (int64_t)kb * GBK;
        return fetch_block(p, n_fixed, kcol, n_fixed < p.wrows);
      } else {
        const int64_t n = (int64_t)kb * GBK + nl;
        return fetch_block(p, n, kcol_fixed, n < p.wrows && kcol_fixed < p.wcols);
      }
    };
    Fetch f0 = fetch_k(0), f1 = fetch_k(1);
    int stage = 0;
    uint32_t ph = 0;
    for (int kb = 0; kb < num_k; ++kb) {
      const Fetch f2 = fetch_k(kb + 2);
      const bool ok = mbar_wait_bounded(empty_bar(stage), ph ^ 1, cta_err, p.status);
      if (ok) dequant_store_row(p, f0, smem0 + stage * SB + kABytes + row_off, swz);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(full_bar(stage));
      f0 = f1;
      f1 = f2;
      if (++stage == S) {
        stage = 0;
        ph ^= 1;
      }
    }

    // ---------------------------------------------------------- epilogue
    mbar_wait_bounded(acc_bar, 0, cta_err, p.status);
    tc_fence_after();
    if (warp < 4) {
      // LoRA down-projection (t or u): save fp32, stage s * aux as bf16.
      const int rl = warp * 32 + lane;
      const int row = m0 + rl;
      const bool save = p.aux_out != nullptr && blockIdx.x == 0 && row < p.M;
      for (int cb = 0; cb < RP / 16; ++cb) {
        uint32_t v[16];
        tmem_ld16(tmem_aux + ((uint32_t)(warp * 32) << 16) + cb * 16, v);
        tmem_ld_wait();
        if (save) {
          for (int j = 0; j < 16; ++j) {
            const int col = cb * 16 + j;
            if (col < p.r) p.aux_out[(int64_t)row * p.r + col] = __uint_as_float(v[j]);
          }
        }
        uint32_t w[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
          w[j] = pack_bf16x2(p.s * __uint_as_float(v[2 * j]), p.s * __uint_as_float(v[2 * j + 1]));
        const uint32_t base = upa_u + cb * (GBM * 32) + (rl >> 3) * 256 + (rl & 7) * 32;
        const uint32_t x = (rl >> 2) & 1;
        sts_v4(base + ((0 ^ x) << 4), w[0], w[1], w[2], w[3]);
        sts_v4(base + ((1 ^ x) << 4), w[4], w[5], w[6], w[7]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(upa_bar);
    }
    mbar_wait_bounded(acc2_bar, 0, cta_err, p.status);
    tc_fence_after();
    const int quarter = warp & 3, half = warp >> 2;
    const int row = m0 + quarter * 32 + lane;
    for (int ch = 0; ch < 4; ++ch) {
      const int col = half * 128 + ch * 32;
      uint32_t v[32];
      tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + col, v);
      tmem_ld_wait();
      const int gcol = c0 + col;
      if (row < p.M && gcol < p.out_cols) {
        const bool full = gcol + 32 <= p.out_cols;
        if (p.out_bf16) {
          uint16_t *dst = reinterpret_cast<uint16_t *>(p.out) + (int64_t)row * p.out_cols + gcol;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            if (full || gcol + 8 * q < p.out_cols) {
              uint4 o;
              o.x = pack_bf16x2(__uint_as_float(v[8 * q + 0]), __uint_as_float(v[8 * q + 1]));
              o.y = pack_bf16x2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3]));
              o.z = pack_bf16x2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5]));
              o.w = pack_bf16x2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7]));
              *reinterpret_cast<uint4 *>(dst + 8 * q) = o;
            }
          }
        } else {
          float *dst = reinterpret_cast<float *>(p.out) + (int64_t)row * p.out_cols + gcol;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            if (full || gcol + 4 * q < p.out_cols)
              *reinterpret_cast<uint4 *>(dst + 4 * q) =
                  make_uint4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
          }
        }
      }
    }
  } else if (warp == 8) {
    // --------------------------------------------------------- TMA producer
    if (lane == 0) {
      const int ncb = RP / 16;
      mbar_arrive_expect_tx(upb_bar, ncb * GBN * 32);
      for (int cb = 0; cb < ncb; ++cb)
        tma_load_2d(upb_u + cb * (GBN * 32), &tmL2, upb_bar, cb * 16, c0);
      int stage = 0;
      uint32_t ph = 0;
      int issued = 0;
      for (int kb = 0; kb < num_k; ++kb) {
        if (!mbar_wait_bounded(empty_bar(stage), ph ^ 1, cta_err, p.status)) break;
        const uint32_t a_dst = smem0 + stage * SB;
        mbar_arrive_expect_tx(full_bar(stage), kABytes + RP * 128);
        tma_load_2d(a_dst, &tmA, full_bar(stage), kb * GBK, m0);
        tma_load_2d(a_dst + kABytes + kBBytes, &tmL1, full_bar(stage), kb * GBK, 0);
        ++issued;
        if (++stage == S) {
          stage = 0;
          ph ^= 1;
        }
      }
      if (*cta_err) {
        // Error path: let every issued copy land before the CTA exits.
        mbar_drain(upb_bar, 0);
        const int first = issued > S ? issued - S : 0;
        for (int i = first; i < issued; ++i) mbar_drain(full_bar(i % S), (i / S) & 1);
      }
    }
    __syncwarp();
  } else {
    // ----------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_main = make_idesc_bf16(GBM, GBN, kDx);
      const uint32_t idesc_aux = make_idesc_bf16(GBM, RP, false);
      constexpr uint32_t idesc_up = make_idesc_bf16(GBM, GBN, false);
      int stage = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int kb = 0; kb < num_k && ok; ++kb) {
        ok = mbar_wait_bounded(full_bar(stage), ph, cta_err, p.status);
        if (!ok) break;
        tc_fence_after();
        const uint32_t a_base = smem0 + stage * SB;
        const uint32_t b_base = a_base + kABytes;
        const uint32_t l_base = b_base + kBBytes;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t ad = make_sdesc(a_base + kk * 32, 16, 1024, kSwz128);
          const uint64_t bd = kDx ? make_sdesc(b_base + kk * 2048, 8192, 1024, kSwz128)
                                  : make_sdesc(b_base + kk * 32, 16, 1024, kSwz128);
          const uint64_t ld = make_sdesc(l_base + kk * 32, 16, 1024, kSwz128);
          const uint32_t accum = (kb > 0 || kk > 0) ? 1u : 0u;
          tc_mma(tmem, ad, bd, idesc_main, accum);
          tc_mma(tmem_aux, ad, ld, idesc_aux, accum);
        }
        tc_commit(empty_bar(stage));
        if (++stage == S) {
          stage = 0;
          ph ^= 1;
        }
      }
      tc_commit(acc_bar);
      if (ok && mbar_wait_bounded(upa_bar, 0, cta_err, p.status) &&
          mbar_wait_bounded(upb_bar, 0, cta_err, p.status)) {
        tc_fence_after();
        for (int cb = 0; cb < RP / 16; ++cb) {
          const uint64_t ad = make_sdesc(upa_u + cb * (GBM * 32), 16, 256, kSwz32);
          const uint64_t bd = make_sdesc(upb_u + cb * (GBN * 32), 16, 256, kSwz32);
          tc_mma(tmem, ad, bd, idesc_up, 1u);
        }
      }
      tc_commit(acc2_bar);
      if (*cta_err) mbar_drain(acc2_bar, 0);  // all issued MMAs retired
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------ host launcher
cudaError_t launch_gemm(bool dx, const CUtensorMap &tmA, const CUtensorMap &tmL1,
                        const CUtensorMap &tmL2, const GemmArgs &args, cudaStream_t s) {
  const int smem = gemm_smem_bytes(args.stages, args.r_pad);
  static bool attr_set[2] = {false, false};
  cudaError_t e;
  if (!attr_set[dx]) {
    if (dx)
      e = cudaFuncSetAttribute(qlora_gemm_kernel<true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
    else
      e = cudaFuncSetAttribute(qlora_gemm_kernel<false>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
    if (e != cudaSuccess) return e;
    attr_set[dx] = true;
  }
  dim3 grid((args.out_cols + GBN - 1) / GBN, (args.M + GBM - 1) / GBM);
  if (dx)
    qlora_gemm_kernel<true><<<grid, kGemmThreads, smem, s>>>(tmA, tmL1, tmL2, args);
  else
    qlora_gemm_kernel<false><<<grid, kGemmThreads, smem, s>>>(tmA, tmL1, tmL2, args);
  return cudaGetLastError();
}

int gemm_pick_stages(int r_pad) {
  for (int st = 4; st >= 2; --st)
    if (gemm_smem_bytes(st, r_pad) <= 232448) return st;
  return 0;
}

}  // namespace qlora
