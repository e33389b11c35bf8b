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
// CTA pairs (a cluster of 2) share one 256 x BN output tile through
// tcgen05 cta_group::2: CTA r owns rows [128r, 128r+128) of the tile and
// half of the B operand (BN/2 output columns); one thread of the leader CTA
// issues every MMA for both.  Contraction step 64.
//
// The kernel is persistent: one cluster per SM pair walks the output tiles
// cid, cid + clusters, ... (row tiles fastest, so the clusters that run at
// the same time share weight columns in L2).  Stage ring positions and
// barrier phases run on across tiles, and TMEM holds two accumulators, so
// the epilogue of one tile overlaps the main loop of the next.
// Per CTA, 704 threads:
//   warps 0-15 dequantising producers in 4 groups that take the stages
//              round-robin; a thread owns one B row of its group's stage and
//              turns its 64 packed nibbles into bf16 through the per-block
//              table T[i] = bf16(c_i * a_hat) indexed with byte permutes; the
//              values go straight into the 128-byte-swizzled operand layout
//              the tensor core reads (K-major forward, MN-major dX).
//   warps 16-19 epilogue: TMEM -> registers -> global, one row per thread.
//   warp 20    TMA: this CTA's 128 activation rows per stage; its halves of
//              the two rank-r LoRA operands once per tile (double-buffered).
//   warp 21    TMEM allocation (both CTAs); in the leader the single MMA
//              issuer, in the peer a relay that forwards "stage ready" to the
//              leader's barriers.
// Per tile the leader first issues r_pad/16 MMAs (256 x BN x 16) for the
// LoRA term, then 4 per stage for the base product, into TMEM columns
// [256 b, 256 b + BN) of both CTAs, b alternating between tiles.
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
constexpr int kEpiWarp0 = kProdWarps;               // 4 epilogue warps (TMEM lane quarters)
constexpr int kTmaWarp = kProdWarps + 4, kMmaWarp = kProdWarps + 5;
constexpr int kGemmThreads = (kProdWarps + 6) * 32;  // 704
constexpr int kAccCols = 256;                        // TMEM columns per accumulator
static_assert(kEpiWarp0 % 4 == 0, "epilogue warp q must own TMEM lane quarter q");
constexpr int kABytes = GBM * GBK * 2;     // 16 KB
constexpr int kBBytes = kHalfN * GBK * 2;  // 16 KB (this CTA's half of B)

__host__ __device__ inline int gemm_stage_bytes(int) { return kABytes + kBBytes; }
__host__ __device__ inline int gemm_upa_bytes(int r_pad) { return (r_pad / 16) * GBM * 32; }
__host__ __device__ inline int gemm_upb_bytes(int r_pad) { return (r_pad / 16) * kHalfN * 32; }
__host__ inline int gemm_smem_bytes(int stages, int r_pad) {
  return 1024 + stages * gemm_stage_bytes(r_pad) +
         2 * (gemm_upa_bytes(r_pad) + gemm_upb_bytes(r_pad)) + 256;
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

// Output tile `tile` of the (row tiles) x (column tiles) grid, row tiles
// fastest.
struct TileSched {
  int mp, total, cid, ncl, count;  // row tiles, tiles, this cluster, clusters, my tiles
  __device__ TileSched(const GemmArgs &p) {
    mp = (p.M + 2 * GBM - 1) / (2 * GBM);
    total = mp * ((p.out_cols + p.bn - 1) / p.bn);
    cid = (int)(blockIdx.x >> 1);
    ncl = (int)(gridDim.x >> 1);
    count = cid < total ? (total - cid + ncl - 1) / ncl : 0;
  }
  __device__ void coords(int it, int &mt, int &nt) const {
    const int tile = cid + it * ncl;
    nt = tile / mp;
    mt = tile - nt * mp;
  }
};

// One producer thread's walk over its group's stages: every 4th position
// of the cluster's stage sequence (tile it, contraction block kb).
struct ProdCursor {
  int it, kb;
  bool live, rowok;
  int64_t q0, b0;  // packed-byte offset / block index of this row's stage 0
};

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
  const int UPA = gemm_upa_bytes(RP), UPB = gemm_upb_bytes(RP);
  uint8_t *upa = smem + S * SB;           // 2 buffers
  uint8_t *upb = upa + 2 * UPA;           // 2 buffers
  uint64_t *bars = reinterpret_cast<uint64_t *>(upb + 2 * UPB);
  // bars: full[S], empty[S], up_full[2], up_empty[2], acc_full[2], acc_empty[2]
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * S + 8);
  const uint32_t cta_err = smem_u32(tmem_slot + 1);  // shared address of the error flag

  const uint32_t smem0 = smem_u32(smem);
  const uint32_t upa_u = smem_u32(upa), upb_u = smem_u32(upb);
  auto full_bar = [&](int s) { return smem_u32(bars + s); };
  auto empty_bar = [&](int s) { return smem_u32(bars + S + s); };
  auto up_full = [&](int b) { return smem_u32(bars + 2 * S + b); };
  auto up_empty = [&](int b) { return smem_u32(bars + 2 * S + 2 + b); };
  auto acc_full = [&](int b) { return smem_u32(bars + 2 * S + 4 + b); };
  auto acc_empty = [&](int b) { return smem_u32(bars + 2 * S + 6 + b); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int BN = p.bn, HN = p.bn / 2;  // pair tile columns / this CTA's B rows
  const int num_k = (p.kdim + GBK - 1) / GBK;
  const TileSched ts(p);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      // TMA arrive + the 4 warps of one producer group (+ the peer's relay)
      mbar_init(full_bar(s), 1 + 4 + (leader ? 1 : 0));
      mbar_init(empty_bar(s), 1);  // multicast tcgen05.commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(up_full(b), 1 + (leader ? 1 : 0));  // TMA arrive (+ the peer's relay)
      mbar_init(up_empty(b), 1);                     // multicast tcgen05.commit
      mbar_init(acc_full(b), 1);                     // multicast tcgen05.commit
      mbar_init(acc_empty(b), leader ? 8 : 1);       // 4 epilogue warps of each CTA
    }
    st_shared_volatile(cta_err, 0u);
    fence_barrier_init();
  }
  if (warp == kTmaWarp && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmL1);
    tma_prefetch_desc(&tmL2);
  }
  if (warp == kMmaWarp) tmem_alloc2(smem_u32(tmem_slot), 2 * kAccCols);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem = ld_shared_volatile(smem_u32(tmem_slot));
  const int total_stages = ts.count * num_k;

  if (warp < kProdWarps) {
    // ------------------------------------------------ dequantising producers
    // Group `grp` (4 warps) produces the cluster's stages g = grp, grp + 4,
    // ...; within a group thread `rowi` owns one 128-byte row of this CTA's
    // B half.
    const int grp = threadIdx.x >> 7;
    const int rowi = threadIdx.x & 127;
    const bool row_used = rowi < HN;  // rows past the pair tile's half are not read
    uint32_t row_off, swz;
    int nl = 0, bsub = 0;
    if (!kDx) {
      row_off = (rowi >> 3) * 1024 + (rowi & 7) * 128;
      swz = rowi & 7;
    } else {
      bsub = rowi >> 6;  // which 64-column atom of this CTA's outputs
      nl = rowi & 63;    // contraction row inside the stage
      row_off = bsub * 8192 + (nl >> 3) * 1024 + (nl & 7) * 128;
      swz = nl & 7;
    }
    // Step per stage (64 contraction elements) of the packed-byte offset and
    // of the block index.
    const int64_t kbr = p.wcols >> 6;  // blocks per weight row
    const int64_t qstep = kDx ? 64 * (p.wcols >> 1) : 32;
    const int64_t bstep = kDx ? 64 * kbr : 1;
    auto set_tile = [&](ProdCursor &c) {
      c.live = c.it < ts.count;
      int mt, nt;
      ts.coords(c.live ? c.it : 0, mt, nt);
      const int64_t cb0 = (int64_t)nt * BN + (int64_t)rank * HN;
      if (!kDx) {
        const int64_t n = cb0 + rowi;  // weight row = output column
        c.rowok = row_used && n < p.wrows;
        c.q0 = n * (p.wcols >> 1);
        c.b0 = n * kbr;
      } else {
        const int64_t kcol = cb0 + 64 * bsub;
        c.rowok = row_used && kcol < p.wcols;
        c.q0 = (int64_t)nl * (p.wcols >> 1) + (kcol >> 1);
        c.b0 = (int64_t)nl * kbr + (kcol >> 6);
      }
    };
    auto advance = [&](ProdCursor &c) {
      c.kb += kProdGroups;
      if (c.kb >= num_k) {
        while (c.kb >= num_k) {
          c.kb -= num_k;
          ++c.it;
        }
        set_tile(c);
      }
    };
    auto fetch = [&](const ProdCursor &c) -> Fetch {
      bool valid = c.live && c.rowok;
      if (kDx) valid = valid && (int64_t)c.kb * GBK + nl < p.wrows;
      return fetch_block(p, valid ? c.q0 + c.kb * qstep : 0, valid ? c.b0 + c.kb * bstep : 0,
                         valid);
    };
    ProdCursor cf;
    cf.it = 0;
    cf.kb = grp;
    while (cf.kb >= num_k) {
      cf.kb -= num_k;
      ++cf.it;
    }
    set_tile(cf);
    // Three-slot ring of prefetched blocks, indexed by compile-time
    // constants only: this group's i-th stage consumes slot i % 3 and
    // refills slot (i + 2) % 3, so no register ever copies a load in flight.
    Fetch f[3];
    f[0] = fetch(cf);
    advance(cf);
    f[1] = fetch(cf);
    advance(cf);
    int stage = grp;
    uint32_t ph = 0;
    while (stage >= S) {
      stage -= S;
      ph ^= 1u;
    }
    for (int g0 = grp; g0 < total_stages; g0 += 3 * kProdGroups) {
#pragma unroll
      for (int u = 0; u < 3; ++u) {
        if (g0 + u * kProdGroups < total_stages) {
          f[(u + 2) % 3] = fetch(cf);
          advance(cf);
          const bool ok = mbar_wait_bounded(empty_bar(stage), ph ^ 1, cta_err, p.status);
          if (ok && row_used) dequant_store_row(p, f[u], smem0 + stage * SB + kABytes + row_off, swz);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(full_bar(stage));
          stage += kProdGroups;
          while (stage >= S) {
            stage -= S;
            ph ^= 1u;
          }
        }
      }
    }
  } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + 4) {
    // ---------------------------------------------------------- epilogue
    // Warp q reads TMEM lanes [32q, 32q + 32): one output row per thread.
    const int quarter = warp & 3;
    for (int it = 0; it < ts.count; ++it) {
      const int b = it & 1;
      const bool ok = mbar_wait_bounded(acc_full(b), (uint32_t)(it >> 1) & 1u, cta_err, p.status);
      tc_fence_after();
      int mt, nt;
      ts.coords(it, mt, nt);
      const int row = mt * (2 * GBM) + (int)rank * GBM + quarter * 32 + lane;
      const int c0 = nt * BN;
      const uint32_t tbase = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(b * kAccCols);
      for (int col = 0; col < BN && ok; col += 32) {
        uint32_t v[32];
        tmem_ld32(tbase + col, v);
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
      // This warp is done reading accumulator b: free it for tile it + 2.
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader)
          mbar_arrive(acc_empty(b));
        else
          mbar_arrive_remote(mapa_shared(acc_empty(b), 0));
      }
    }
  } else if (warp == kTmaWarp) {
    // --------------------------------------------------------- TMA producer
    if (lane == 0) {
      const int ncb = RP / 16;
      // LoRA operand halves of tile j into buffer j & 1, one tile ahead.
      auto issue_up = [&](int j) {
        const int b = j & 1;
        if (!mbar_wait_bounded(up_empty(b), ((uint32_t)(j >> 1) & 1u) ^ 1u, cta_err, p.status))
          return false;
        int mt, nt;
        ts.coords(j, mt, nt);
        const int m0 = mt * (2 * GBM) + (int)rank * GBM;
        const int cb0 = nt * BN + (int)rank * HN;
        mbar_arrive_expect_tx(up_full(b), ncb * (GBM + HN) * 32);
        for (int cb = 0; cb < ncb; ++cb) {
          tma_load_2d(upa_u + b * UPA + cb * (GBM * 32), &tmL1, up_full(b), cb * 16, m0);
          tma_load_2d(upb_u + b * UPB + cb * (kHalfN * 32), &tmL2, up_full(b), cb * 16, cb0);
        }
        return true;
      };
      int stage = 0;
      uint32_t ph = 0;
      int issued = 0, up_issued = 0;
      bool ok = true;
      for (int it = 0; it < ts.count && ok; ++it) {
        if (it == 0) {
          ok = issue_up(0);
          up_issued += ok;
        }
        if (ok && it + 1 < ts.count) {
          ok = issue_up(it + 1);
          up_issued += ok;
        }
        int mt, nt;
        ts.coords(it, mt, nt);
        const int m0 = mt * (2 * GBM) + (int)rank * GBM;
        for (int kb = 0; kb < num_k && ok; ++kb) {
          ok = mbar_wait_bounded(empty_bar(stage), ph ^ 1, cta_err, p.status);
          if (!ok) break;
          mbar_arrive_expect_tx(full_bar(stage), kABytes);
          tma_load_2d(smem0 + stage * SB, &tmA, full_bar(stage), kb * GBK, m0);
          ++issued;
          if (++stage == S) {
            stage = 0;
            ph ^= 1;
          }
        }
      }
      if (ld_shared_volatile(cta_err)) {
        // Error path: let every issued copy land before the CTA exits.
        for (int j = up_issued > 2 ? up_issued - 2 : 0; j < up_issued; ++j)
          mbar_drain(up_full(j & 1), (uint32_t)(j >> 1) & 1u);
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
      int stage = 0;
      uint32_t ph = 0;
      bool ok = true;
      int last_acc = -1;
      for (int it = 0; it < ts.count && ok; ++it) {
        const int b = it & 1;
        const uint32_t use_ph = (uint32_t)(it >> 1) & 1u;
        ok = mbar_wait_bounded(acc_empty(b), use_ph ^ 1u, cta_err, p.status);
        if (ok) ok = mbar_wait_bounded(up_full(b), use_ph, cta_err, p.status);
        if (!ok) break;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(b * kAccCols);
        // LoRA term first: D = (s.t) . B^T  (or (s.u) . A for dX)
        for (int cb = 0; cb < RP / 16; ++cb) {
          const uint64_t ad = make_sdesc(upa_u + b * UPA + cb * (GBM * 32), 16, 256, kSwz32);
          const uint64_t bd = make_sdesc(upb_u + b * UPB + cb * (kHalfN * 32), 16, 256, kSwz32);
          tc_mma2(d, ad, bd, idesc_up, cb > 0 ? 1u : 0u);
        }
        tc_commit2_mc(up_empty(b), 0x3);
        for (int kb = 0; kb < num_k; ++kb) {
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
            tc_mma2(d, ad, bd, idesc_main, 1u);
          }
          tc_commit2_mc(empty_bar(stage), 0x3);
          if (++stage == S) {
            stage = 0;
            ph ^= 1;
          }
        }
        tc_commit2_mc(acc_full(b), 0x3);
        last_acc = it;
      }
      // Error path: every issued MMA retired before TMEM is freed.
      if (ld_shared_volatile(cta_err) && last_acc >= 0)
        mbar_drain(acc_full(last_acc & 1), (uint32_t)(last_acc >> 1) & 1u);
    }
    __syncwarp();
  } else {
    // ----------------------------------------------- relay (peer CTA)
    // Forwards, per tile, "this CTA's LoRA operand halves landed" and then,
    // per stage, "this CTA's half of stage s is ready" (its TMA bytes landed
    // and the 4 warps of the producer group arrived) to the leader's
    // barriers, in the order the leader consumes them.
    if (lane == 0) {
      int stage = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int it = 0; it < ts.count && ok; ++it) {
        const int b = it & 1;
        ok = mbar_wait_bounded(up_full(b), (uint32_t)(it >> 1) & 1u, cta_err, p.status);
        if (!ok) break;
        mbar_arrive_remote(mapa_shared(up_full(b), 0));
        for (int kb = 0; kb < num_k; ++kb) {
          ok = mbar_wait_bounded(full_bar(stage), ph, cta_err, p.status);
          if (!ok) break;
          mbar_arrive_remote(mapa_shared(full_bar(stage), 0));
          if (++stage == S) {
            stage = 0;
            ph ^= 1;
          }
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
    tmem_dealloc2(tmem, 2 * kAccCols);
  }
}

// ------------------------------------------------------------ host launcher
cudaError_t launch_gemm(bool dx, const CUtensorMap &tmA, const CUtensorMap &tmL1,
                        const CUtensorMap &tmL2, const GemmArgs &args, cudaStream_t s) {
  const int smem = gemm_smem_bytes(args.stages, args.r_pad);
  static bool attr_set[2] = {false, false};
  // Clusters that fit on the device at once, per (kernel, shared memory size).
  static int cached_clusters[2] = {0, 0}, cached_smem[2] = {-1, -1}, cached_dev[2] = {-1, -1};
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
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if (cached_smem[dx] != smem || cached_dev[dx] != dev) {
    int n = 0;
    cfg.gridDim = dim3(2, 1, 1);
    if (dx)
      e = cudaOccupancyMaxActiveClusters(&n, qlora_gemm_kernel<true>, &cfg);
    else
      e = cudaOccupancyMaxActiveClusters(&n, qlora_gemm_kernel<false>, &cfg);
    if (e != cudaSuccess) return e;
    if (n < 1) return cudaErrorInvalidConfiguration;
    cached_clusters[dx] = n;
    cached_smem[dx] = smem;
    cached_dev[dx] = dev;
  }
  const long tiles = (long)((args.M + 2 * GBM - 1) / (2 * GBM)) *
                     ((args.out_cols + args.bn - 1) / args.bn);
  if (tiles == 0) return cudaSuccess;
  const int clusters = (int)(tiles < cached_clusters[dx] ? tiles : cached_clusters[dx]);
  cfg.gridDim = dim3(2 * clusters, 1, 1);
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
