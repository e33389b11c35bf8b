// gemm_tc.cu -- fused dequantise + tcgen05 GEMM + LoRA bypass for sm_103a.
//
// One kernel serves both dense contractions of the QLoRA linear layer
// ("QLoRA and 4bit Quantization | QLoRA 与 4-bit 量化", Step 3 formula and the
// gradient routing of Step 4's frozen-base test):
//   forward  (kDx = false): out[M, N] = (s.t)[M, r] . B[N, r]^T + x[M, K] . W_hat[N, K]^T
//   backward (kDx = true) : out[M, K] = (s.u)[M, r] . A^T[K, r]^T + dY[M, N] . W_hat[N, K]
// where t = x A^T (u = dY B) comes in as bf16(s.t) from a small tensor-core
// pre-pass (lora_grad.cu) and seeds the accumulator before the main loop.
//
// CTA pairs (a cluster of 2) share one 256 x 256 output tile through
// tcgen05 cta_group::2: CTA r owns rows [128r, 128r+128) of the tile and
// half of the B operand (output columns [128r, 128r+128)); one thread of the
// leader CTA issues every MMA for both.  Contraction step 64.
// Per CTA, 576 threads:
//   warps 0-15 dequantising producers in 4 groups that take the stages
//              round-robin; a thread owns one B row of its group's stage and
//              turns its 64 packed nibbles into bf16 through the per-block
//              table T[i] = bf16(c_i * a_hat) indexed with byte permutes; the
//              values go straight into the 128-byte-swizzled operand layout
//              the tensor core reads (K-major forward, MN-major dX).  After
//              the main loop the same warps run the epilogue.
//   warp 16    TMA: this CTA's 128 activation rows per stage; its halves of
//              the two rank-r LoRA operands once.
//   warp 17    TMEM allocation (both CTAs); in the leader the single MMA
//              issuer, in the peer a relay that forwards "stage ready" to the
//              leader's barrier.
// The leader first issues r_pad/16 MMAs (256 x 256 x 16) for the LoRA term,
// then 4 per stage for the base product, all into TMEM columns [0, 256) of
// both CTAs; the epilogue moves TMEM -> registers -> global.
//
// Each SM dequantises 128 x 64 weights per stage for 2 x 128 x 256 x 64
// MMA work, half of what a single-CTA 128 x 256 tile needs; the integer
// pipe that runs the byte permutes is the resource this saves.
//
// Every mbarrier wait is bounded (common.cuh): a wait that runs out writes
// QLORA_ERR_TIMEOUT to the device status word and every role runs to the
// end of the kernel without blocking.
#include "common.cuh"
#include "kernels.h"

namespace qlora {

constexpr int GBM = 128;  // rows per CTA (the pair covers 256)
constexpr int GBN = 256;  // output columns per pair tile
constexpr int GBK = 64;
constexpr int kHalfN = GBN / 2;
constexpr int kProdGroups = 4;                     // producer groups, stages round-robin
constexpr int kProdWarps = 4 * kProdGroups;        // 16 warps: one thread per B row per group
constexpr int kTmaWarp = kProdWarps, kMmaWarp = kProdWarps + 1;
constexpr int kGemmThreads = (kProdWarps + 2) * 32;  // 576
constexpr int kABytes = GBM * GBK * 2;     // 16 KB
constexpr int kBBytes = kHalfN * GBK * 2;  // 16 KB (this CTA's half of B)

__host__ __device__ inline int gemm_stage_bytes(int) { return kABytes + kBBytes; }
__host__ __device__ inline int gemm_upa_bytes(int r_pad) { return (r_pad / 16) * GBM * 32; }
__host__ __device__ inline int gemm_upb_bytes(int r_pad) { return (r_pad / 16) * kHalfN * 32; }
__host__ inline int gemm_smem_bytes(int stages, int r_pad) {
  return 1024 + stages * gemm_stage_bytes(r_pad) + gemm_upa_bytes(r_pad) + gemm_upb_bytes(r_pad) +
         256;
}

// Raw packed bytes + block constant of one 64-block.
// Loaded values stay raw until use: converting a value right after its load
// would stall the thread for the whole load latency at prefetch time.
struct Fetch {
  uint4 lo, hi;  // 32 packed bytes
  int code;  // int8 block constant (DQ)
  float c;   // second-level scale s2 (DQ) or fp32 absmax (no DQ)
  bool valid;
};

// Loads are unconditional (the caller clamps the address into range).
// `qoff` is the byte offset of the 32 packed bytes, `blk` the block index.
__device__ __forceinline__ Fetch fetch_block(const GemmArgs &p, int64_t qoff, int64_t blk,
                                            bool valid) {
  Fetch f;
  f.valid = valid;
  f.lo = ldg_nc_v4(p.packed + qoff);
  f.hi = ldg_nc_v4(p.packed + qoff + 16);
  f.code = ldg_nc_s8(p.codes + (p.use_code ? blk : 0));
  f.c = ldg_nc_f32(p.cvec + (blk >> p.cshift));
  return f;
}

// Dequantise one 64-block into the 8 16-byte chunks of one 128-byte
// swizzled row at `row_addr` (chunk c goes to position c ^ swz).
__device__ __forceinline__ void dequant_store_row(const GemmArgs &p, const Fetch &f,
                                                  uint32_t row_addr, uint32_t swz) {
  if (!f.valid) {
#pragma unroll
    for (int c = 0; c < 8; ++c) sts_v4(row_addr + ((c ^ swz) << 4), 0, 0, 0, 0);
    return;
  }
  const float ahat = p.use_code ? __fmul_rn((float)f.code, f.c) : f.c;
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
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * S + 2);
  const uint32_t cta_err = smem_u32(tmem_slot + 1);  // shared address of the error flag

  const uint32_t smem0 = smem_u32(smem);
  const uint32_t upa_u = smem_u32(upa), upb_u = smem_u32(upb);
  auto full_bar = [&](int s) { return smem_u32(bars + s); };
  auto empty_bar = [&](int s) { return smem_u32(bars + S + s); };
  const uint32_t up_bar = smem_u32(bars + 2 * S);
  const uint32_t acc_bar = smem_u32(bars + 2 * S + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int m0 = (blockIdx.x >> 1) * (2 * GBM) + (int)rank * GBM;  // this CTA's rows
  const int BN = p.bn, HN = p.bn / 2;  // pair tile columns / this CTA's B rows
  const int c0 = blockIdx.y * BN;                                  // pair's output columns
  const int cb0 = c0 + (int)rank * HN;                             // this CTA's B half
  const int num_k = (p.kdim + GBK - 1) / GBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      // TMA arrive + the 4 warps of one producer group (+ the peer's relay)
      mbar_init(full_bar(s), 1 + 4 + (leader ? 1 : 0));
      mbar_init(empty_bar(s), 1);  // multicast tcgen05.commit
    }
    mbar_init(up_bar, 1 + (leader ? 1 : 0));  // TMA arrive (+ the peer's relay)
    mbar_init(acc_bar, 1);
    st_shared_volatile(cta_err, 0u);
    fence_barrier_init();
  }
  if (warp == kTmaWarp && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmL1);
    tma_prefetch_desc(&tmL2);
  }
  if (warp == kMmaWarp) tmem_alloc2(smem_u32(tmem_slot), 256);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem = ld_shared_volatile(smem_u32(tmem_slot));

  if (warp < kProdWarps) {
    // ------------------------------------------------ dequantising producers
    // Group `grp` (4 warps) produces stages kb = grp, grp + 4, ...; within a
    // group thread `rowi` owns one 128-byte row of this CTA's B half.
    const int grp = threadIdx.x >> 7;
    const int rowi = threadIdx.x & 127;
    int64_t n_fixed = 0, kcol_fixed = 0;
    uint32_t row_off, swz;
    int nl = 0;
    if (!kDx) {
      n_fixed = (int64_t)cb0 + rowi;  // weight row = output column
      row_off = (rowi >> 3) * 1024 + (rowi & 7) * 128;
      swz = rowi & 7;
    } else {
      const int bsub = rowi >> 6;  // which 64-column atom of this CTA's 128 outputs
      nl = rowi & 63;              // contraction row inside the stage
      kcol_fixed = (int64_t)cb0 + 64 * bsub;
      row_off = bsub * 8192 + (nl >> 3) * 1024 + (nl & 7) * 128;
      swz = nl & 7;
    }
    // Byte offset / block index of this thread's 32 packed bytes at stage 0
    // and their step per stage (64 contraction elements).
    const int64_t kbr = p.wcols >> 6;  // blocks per weight row
    int64_t q0, b0, qstep, bstep;
    if (!kDx) {
      q0 = n_fixed * (p.wcols >> 1);  // row n, columns [0, 64)
      b0 = n_fixed * kbr;
      qstep = 32;
      bstep = 1;
    } else {
      q0 = (int64_t)nl * (p.wcols >> 1) + (kcol_fixed >> 1);
      b0 = (int64_t)nl * kbr + (kcol_fixed >> 6);
      qstep = 64 * (p.wcols >> 1);
      bstep = 64 * kbr;
    }
    const bool row_used = rowi < HN;  // rows past the pair tile's half are not read
    auto fetch_k = [&](int kb) -> Fetch {
      const bool in_k = kb < num_k;
      const int kbc = in_k ? kb : num_k - 1;
      bool valid;
      if (!kDx)
        valid = in_k && row_used && n_fixed < p.wrows;
      else
        valid = in_k && row_used && (int64_t)kbc * GBK + nl < p.wrows && kcol_fixed < p.wcols;
      return fetch_block(p, valid ? q0 + kbc * qstep : 0, valid ? b0 + kbc * bstep : 0, valid);
    };
    // Three-slot ring of prefetched blocks, indexed by compile-time
    // constants only: this group's i-th stage consumes slot i % 3 and
    // refills slot (i + 2) % 3, so no register ever copies a load in flight.
    Fetch f[3];
    f[0] = fetch_k(grp);
    f[1] = fetch_k(grp + kProdGroups);
    for (int kb0 = grp; kb0 < num_k; kb0 += 3 * kProdGroups) {
#pragma unroll
      for (int u = 0; u < 3; ++u) {
        const int kb = kb0 + u * kProdGroups;
        if (kb < num_k) {
          f[(u + 2) % 3] = fetch_k(kb + 2 * kProdGroups);
          const int stage = kb % S;
          const uint32_t ph = (uint32_t)(kb / S) & 1u;
          const bool ok = mbar_wait_bounded(empty_bar(stage), ph ^ 1, cta_err, p.status);
          if (ok && row_used) dequant_store_row(p, f[u], smem0 + stage * SB + kABytes + row_off, swz);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(full_bar(stage));
        }
      }
    }

    // ---------------------------------------------------------- epilogue
    mbar_wait_bounded(acc_bar, 0, cta_err, p.status);
    tc_fence_after();
    // 16 warps: warp w reads TMEM lanes 32*(w%4).. and columns [64*(w/4), +64) of BN
    const int quarter = warp & 3, hcol = warp >> 2;
    const int row = m0 + quarter * 32 + lane;
    for (int ch = 0; ch < 2; ++ch) {
      const int col = hcol * 64 + ch * 32;
      if (col >= BN) break;  // warp-uniform
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
  } else if (warp == kTmaWarp) {
    // --------------------------------------------------------- TMA producer
    if (lane == 0) {
      const int ncb = RP / 16;
      mbar_arrive_expect_tx(up_bar, ncb * (GBM + HN) * 32);
      for (int cb = 0; cb < ncb; ++cb) {
        tma_load_2d(upa_u + cb * (GBM * 32), &tmL1, up_bar, cb * 16, m0);
        tma_load_2d(upb_u + cb * (kHalfN * 32), &tmL2, up_bar, cb * 16, cb0);
      }
      int stage = 0;
      uint32_t ph = 0;
      int issued = 0;
      for (int kb = 0; kb < num_k; ++kb) {
        if (!mbar_wait_bounded(empty_bar(stage), ph ^ 1, cta_err, p.status)) break;
        const uint32_t a_dst = smem0 + stage * SB;
        mbar_arrive_expect_tx(full_bar(stage), kABytes);
        tma_load_2d(a_dst, &tmA, full_bar(stage), kb * GBK, m0);
        ++issued;
        if (++stage == S) {
          stage = 0;
          ph ^= 1;
        }
      }
      if (ld_shared_volatile(cta_err)) {
        // Error path: let every issued copy land before the CTA exits.
        mbar_drain(up_bar, 0);
        const int first = issued > S ? issued - S : 0;
        for (int i = first; i < issued; ++i) mbar_drain(full_bar(i % S), (i / S) & 1);
      }
    }
    __syncwarp();
  } else if (leader) {
    // ------------------------------------------------- MMA issuer (leader)
    if (lane == 0) {
      const uint32_t idesc_main = make_idesc_bf16(2 * GBM, BN, kDx);
      const uint32_t idesc_up = make_idesc_bf16(2 * GBM, BN, false);
      bool ok = mbar_wait_bounded(up_bar, 0, cta_err, p.status);
      if (ok) {
        // LoRA term first: D = (s.t) . B^T  (or (s.u) . A for dX)
        tc_fence_after();
        for (int cb = 0; cb < RP / 16; ++cb) {
          const uint64_t ad = make_sdesc(upa_u + cb * (GBM * 32), 16, 256, kSwz32);
          const uint64_t bd = make_sdesc(upb_u + cb * (kHalfN * 32), 16, 256, kSwz32);
          tc_mma2(tmem, ad, bd, idesc_up, cb > 0 ? 1u : 0u);
        }
      }
      int stage = 0;
      uint32_t ph = 0;
      for (int kb = 0; kb < num_k && ok; ++kb) {
        ok = mbar_wait_bounded(full_bar(stage), ph, cta_err, p.status);
        if (!ok) break;
        tc_fence_after();
        const uint32_t a_base = smem0 + stage * SB;
        const uint32_t b_base = a_base + kABytes;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t ad = make_sdesc(a_base + kk * 32, 16, 1024, kSwz128);
          const uint64_t bd = kDx ? make_sdesc(b_base + kk * 2048, 8192, 1024, kSwz128)
                                  : make_sdesc(b_base + kk * 32, 16, 1024, kSwz128);
          tc_mma2(tmem, ad, bd, idesc_main, 1u);
        }
        tc_commit2_mc(empty_bar(stage), 0x3);
        if (++stage == S) {
          stage = 0;
          ph ^= 1;
        }
      }
      tc_commit2_mc(acc_bar, 0x3);
      if (ld_shared_volatile(cta_err)) mbar_drain(acc_bar, 0);  // all issued MMAs retired
    }
    __syncwarp();
  } else {
    // ----------------------------------------------- relay (peer CTA)
    // Forwards "this CTA's LoRA operand halves landed" and then, per stage,
    // "this CTA's half of stage s is ready" (its TMA bytes landed and the 4
    // warps of the producer group arrived) to the leader's barriers, in the order the
    // leader consumes them.
    if (lane == 0) {
      if (mbar_wait_bounded(up_bar, 0, cta_err, p.status)) mbar_arrive_remote(mapa_shared(up_bar, 0));
      int stage = 0;
      uint32_t ph = 0;
      for (int kb = 0; kb < num_k; ++kb) {
        if (!mbar_wait_bounded(full_bar(stage), ph, cta_err, p.status)) break;
        mbar_arrive_remote(mapa_shared(full_bar(stage), 0));
        if (++stage == S) {
          stage = 0;
          ph ^= 1;
        }
      }
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the pair is done with TMEM and with each other's smem
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc2(tmem, 256);
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
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * ((args.M + 2 * GBM - 1) / (2 * GBM)), (args.out_cols + args.bn - 1) / args.bn, 1);
  cfg.blockDim = dim3(kGemmThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = 2;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  if (dx)
    e = cudaLaunchKernelEx(&cfg, qlora_gemm_kernel<true>, tmA, tmL1, tmL2, args);
  else
    e = cudaLaunchKernelEx(&cfg, qlora_gemm_kernel<false>, tmA, tmL1, tmL2, args);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Pair-tile width: the candidate minimising (waves of tiles over the CTA
// pairs) x (tile width + a fixed per-tile cost of ~40 columns).  The dX
// operand is MN-major in 64-column atoms per CTA, so there only 128 or 256.
int gemm_pick_bn(int M, int out_cols, bool dx, int num_sms) {
  static const int fwd_c[] = {256, 224, 192, 160, 128};
  static const int dx_c[] = {256, 128};
  const int *c = dx ? dx_c : fwd_c;
  const int nc = dx ? 2 : 5;
  const int pairs = num_sms / 2 > 0 ? num_sms / 2 : 1;
  const int mp = (M + 2 * GBM - 1) / (2 * GBM);
  int best = 256;
  long best_cost = -1;
  for (int i = 0; i < nc; ++i) {
    const long tiles = (long)mp * ((out_cols + c[i] - 1) / c[i]);
    const long waves = (tiles + pairs - 1) / pairs;
    const long cost = waves * (c[i] + 40);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = c[i];
    }
  }
  return best;
}

int gemm_pick_stages(int r_pad) {
  for (int st = 7; st >= 2; --st)
    if (gemm_smem_bytes(st, r_pad) <= 232448) return st;
  return 0;
}

}  // namespace qlora
