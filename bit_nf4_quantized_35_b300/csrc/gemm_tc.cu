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
// Per CTA, 704 threads (22 warps; the role table below places them on the
// SM's schedulers):
//   16 dequantising producer warps in 4 groups that take the stages
//              round-robin; a thread owns one B row of its group's stage and
//              turns its 64 packed nibbles into bf16 through the per-block
//              table T[i] = bf16(c_i * a_hat) indexed with byte permutes; the
//              values go straight into the 128-byte-swizzled operand layout
//              the tensor core reads (K-major forward, MN-major dX).
//   4 epilogue warps: TMEM -> registers -> a staging tile in shared memory
//              -> row-contiguous global stores (or, for part of a split
//              tile, fp32 partial sums; see the work schedule below).
//   TMA warp:  this CTA's 128 activation rows per stage; its halves of the
//              two rank-r LoRA operands once per tile (double-buffered).
//   MMA warp:  TMEM allocation (both CTAs); in the leader the single MMA
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
constexpr int kGemmThreads = (kProdWarps + 6) * 32;  // 704
constexpr int kAccCols = 256;                        // TMEM columns per accumulator
// Warp roles.  A warp runs on scheduler (warp index mod 4) of the SM.  The
// MMA issuer and the TMA warp sit on scheduler 3 with one epilogue warp and
// only 2 of the 16 dequantising producers, so the one thread that issues
// every MMA is not starved of issue slots by the producers' integer work
// (the other schedulers carry 4 or 5 producers each).
//   epilogue: warps 0, 1, 2, 11 (TMEM lane quarter = warp mod 4)
//   MMA / relay: warp 3;  TMA: warp 7;  producers: the other 16 warps.
constexpr int kMmaWarp = 3, kTmaWarp = 7, kEpiWarp3 = 11;
__device__ __forceinline__ bool is_epi_warp(int w) { return w < 3 || w == kEpiWarp3; }
__device__ __forceinline__ bool is_prod_warp(int w) {
  return w > 3 && w != kTmaWarp && w != kEpiWarp3;
}
// Producer index 0..15 of producer warp w.
__device__ __forceinline__ int prod_index(int w) {
  return w - 4 - (w > kTmaWarp ? 1 : 0) - (w > kEpiWarp3 ? 1 : 0);
}
static_assert(kEpiWarp3 % 4 == 3 && kMmaWarp % 4 == 3 && kTmaWarp % 4 == 3,
              "roles sharing the MMA issuer's scheduler");
constexpr int kABytes = GBM * GBK * 2;     // 16 KB
constexpr int kBBytes = kHalfN * GBK * 2;  // 16 KB (this CTA's half of B)

__host__ __device__ inline int gemm_stage_bytes(int) { return kABytes + kBBytes; }
__host__ __device__ inline int gemm_upa_bytes(int r_pad) { return (r_pad / 16) * GBM * 32; }
__host__ __device__ inline int gemm_upb_bytes(int r_pad) { return (r_pad / 16) * kHalfN * 32; }
// Epilogue staging: per epilogue warp 32 rows x 16 fp32 columns, row pitch
// 80 bytes (16-byte accesses by 8 consecutive rows hit distinct banks).
constexpr int kStagePitch = 80;
constexpr int kStageWarpBytes = 32 * kStagePitch;  // 2560
constexpr int kStageBytes = 4 * kStageWarpBytes;   // 10 KB
__host__ inline int gemm_smem_bytes(int stages, int r_pad) {
  return 1024 + stages * gemm_stage_bytes(r_pad) +
         2 * (gemm_upa_bytes(r_pad) + gemm_upb_bytes(r_pad)) + kStageBytes + 256;
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
// `qoff` is the byte offset of the 32 packed bytes, `chunk` the index of
// their 64-element chunk of the flattened weight; the chunk lies in block
// chunk >> bshift (block = 64 << bshift elements).
__device__ __forceinline__ Fetch fetch_block(const GemmArgs &p, int64_t qoff, int64_t chunk,
                                            bool valid) {
  Fetch f;
  f.valid = valid;
  f.lo = ldg_nc_v4(p.packed + qoff);
  f.hi = ldg_nc_v4(p.packed + qoff + 16);
  const int64_t blk = chunk >> p.bshift;
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
  const Nf4Table t = make_table(ahat, p.cb);
  const uint32_t w[8] = {f.lo.x, f.lo.y, f.lo.z, f.lo.w, f.hi.x, f.hi.y, f.hi.z, f.hi.w};
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    uint32_t o[4];
    lookup8(t, w[c], o);
    sts_v4(row_addr + ((c ^ swz) << 4), o[0], o[1], o[2], o[3]);
  }
}

// Work schedule.  A unit is one 64-wide contraction block of one output
// tile; tiles are numbered row tiles fastest and a tile's units are
// consecutive.  Cluster c takes units [ubeg(c), ubeg(c + 1)): an equal share
// (the first U % C clusters one more) when tiles are split (sk), else whole
// tiles shared out the same way.  A cluster's range falls into segments at
// tile boundaries; only its first and last segment can be part of a tile,
// and a tile shared by clusters c_first..c_last is finished by whichever of
// them ends last.  All counts fit in 32 bits (the launcher checks U).
struct Sched {
  int mp, num_k, C, c, T, U, u0, u1;
  int q, rr;  // share per cluster and remainder, in units (sk) or tiles
  bool sk;
  __device__ Sched(const GemmArgs &p) {
    mp = (p.M + 2 * GBM - 1) / (2 * GBM);
    num_k = (p.kdim + GBK - 1) / GBK;
    T = mp * ((p.out_cols + p.bn - 1) / p.bn);
    U = T * num_k;
    C = (int)(gridDim.x >> 1);
    c = (int)(blockIdx.x >> 1);
    sk = p.sk != 0;
    const int n = sk ? U : T;
    q = n / C;
    rr = n - q * C;
    u0 = ubeg(c);
    u1 = ubeg(c + 1);
  }
  __device__ int ubeg(int cc) const {
    const int v = cc * q + (cc < rr ? cc : rr);
    return sk ? v : v * num_k;
  }
  // The cluster whose range holds unit u (split mode; q >= 1).
  __device__ int owner(int u) const {
    const int big = rr * (q + 1);
    return u < big ? u / (q + 1) : rr + (u - big) / q;
  }
  __device__ void coords(int t, int &mt, int &nt) const {
    nt = t / mp;
    mt = t - nt * mp;
  }
};

// One segment of a cluster's range: tile t, contraction blocks [kb0, kb1).
struct Seg {
  int t, kb0, kb1;
};
__device__ __forceinline__ Seg seg_at(const Sched &sc, int u) {
  Seg g;
  g.t = u / sc.num_k;
  g.kb0 = u - g.t * sc.num_k;
  const int e = sc.u1 - g.t * sc.num_k;
  g.kb1 = e < sc.num_k ? e : sc.num_k;
  return g;
}

// One producer thread's walk over its group's stages: every 4th unit of the
// cluster's range.
struct ProdCursor {
  int rem;  // units left in the cluster's range from this one on
  int t, kb;
  bool live, rowok;
  int64_t q0, b0;  // packed-byte offset / block index of this row's contraction block 0
};

__device__ __forceinline__ void named_bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
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
  const int UPA = gemm_upa_bytes(RP), UPB = gemm_upb_bytes(RP);
  uint8_t *upa = smem + S * SB;           // 2 buffers
  uint8_t *upb = upa + 2 * UPA;           // 2 buffers
  uint8_t *epi_stage = upb + 2 * UPB;     // 4 x kStageWarpBytes
  uint64_t *bars = reinterpret_cast<uint64_t *>(epi_stage + kStageBytes);
  // bars: full[S], empty[S], up_full[2], up_empty[2], acc_full[2], acc_empty[2]
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * S + 8);
  const uint32_t cta_err = smem_u32(tmem_slot + 1);  // shared address of the error flag
  volatile int *last_flag = reinterpret_cast<volatile int *>(tmem_slot + 2);

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
  const Sched sc(p);
  const int num_k = sc.num_k;

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
  const int total_stages = sc.u1 - sc.u0;
  // Everything above is on-chip set-up; every global access comes after the
  // previous kernel on the stream has completed (programmatic dependent
  // launch).  Dependents are released when this CTA's work is done.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  if (is_prod_warp(warp)) {
    // ------------------------------------------------ dequantising producers
    // Group `grp` (4 warps) produces the cluster's stages g = grp, grp + 4,
    // ...; within a group thread `rowi` owns one 128-byte row of this CTA's
    // B half.
    const int pi = prod_index(warp);
    const int grp = pi >> 2;
    const int rowi = (pi & 3) * 32 + lane;
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
    // Step per contraction block (64 elements) of the packed-byte offset
    // and of the block index.
    const int64_t kbr = p.wcols >> 6;  // blocks per weight row
    const int64_t qstep = kDx ? 64 * (p.wcols >> 1) : 32;
    const int64_t bstep = kDx ? 64 * kbr : 1;
    auto set_tile = [&](ProdCursor &c) {
      int mt, nt;
      sc.coords(c.live ? c.t : 0, mt, nt);
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
      c.rem -= kProdGroups;
      c.kb += kProdGroups;
      c.live = c.rem > 0;
      if (c.kb >= num_k) {
        while (c.kb >= num_k) {
          c.kb -= num_k;
          ++c.t;
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
    {
      const int u = sc.u0 + grp;
      cf.t = u / num_k;
      cf.kb = u - cf.t * num_k;
      cf.rem = sc.u1 - u;
      cf.live = cf.rem > 0;
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
  } else if (is_epi_warp(warp)) {
    // ---------------------------------------------------------- epilogue
    // Warp q reads TMEM lanes [32q, 32q + 32): one output row per thread.
    const int quarter = warp & 3;
    const int ltid = quarter * 32 + lane;  // row within the CTA's 128
    const int first_tile = sc.u0 / num_k;
    int it = 0;
    for (int u = sc.u0; u < sc.u1; ++it) {
      const Seg sg = seg_at(sc, u);
      u = sg.t * num_k + sg.kb1;
      const int b = it & 1;
      const bool ok = mbar_wait_bounded(acc_full(b), (uint32_t)(it >> 1) & 1u, cta_err, p.status);
      tc_fence_after();
      int mt, nt;
      sc.coords(sg.t, mt, nt);
      const int c0 = nt * BN;
      const uint32_t tbase = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(b * kAccCols);
      const bool whole = sg.kb0 == 0 && sg.kb1 == num_k;
      // Output of 16 columns [gcol, gcol + 16) of this warp's 32 rows: each
      // thread puts its row into the warp's staging tile, then the warp
      // writes the tile out row-contiguously (8 rows x 64 bytes per fp32
      // store, 16 rows x 32 bytes per bf16 store).  Output columns are a
      // multiple of 8, so a 4- or 8-column piece is wholly inside or outside.
      const uint32_t stg = smem_u32(epi_stage) + quarter * kStageWarpBytes;
      const int row0 = mt * (2 * GBM) + (int)rank * GBM + quarter * 32;
      auto store_out = [&](int gcol, const float (&a)[16]) {
        __syncwarp();  // the previous chunk's reads of the staging tile are done
        if (p.out_bf16) {
          const uint32_t d = stg + lane * kStagePitch;
          sts_v4(d, pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]), pack_bf16x2(a[4], a[5]),
                 pack_bf16x2(a[6], a[7]));
          sts_v4(d + 16, pack_bf16x2(a[8], a[9]), pack_bf16x2(a[10], a[11]),
                 pack_bf16x2(a[12], a[13]), pack_bf16x2(a[14], a[15]));
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int id = i * 32 + lane, rr = id >> 1, c8 = id & 1;
            const int grow = row0 + rr, gc = gcol + 8 * c8;
            const uint4 w = lds_v4(stg + rr * kStagePitch + c8 * 16);
            if (grow < p.M && gc < p.out_cols)
              *reinterpret_cast<uint4 *>(reinterpret_cast<uint16_t *>(p.out) +
                                         (int64_t)grow * p.out_cols + gc) = w;
          }
        } else {
          const uint32_t d = stg + lane * kStagePitch;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            sts_v4(d + 16 * j, __float_as_uint(a[4 * j]), __float_as_uint(a[4 * j + 1]),
                   __float_as_uint(a[4 * j + 2]), __float_as_uint(a[4 * j + 3]));
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int id = i * 32 + lane, rr = id >> 2, c4 = id & 3;
            const int grow = row0 + rr, gc = gcol + 4 * c4;
            const uint4 w = lds_v4(stg + rr * kStagePitch + c4 * 16);
            if (grow < p.M && gc < p.out_cols)
              *reinterpret_cast<uint4 *>(reinterpret_cast<float *>(p.out) +
                                         (int64_t)grow * p.out_cols + gc) = w;
          }
        }
      };
      // Split-tile slot of 128 rows x 256 columns, laid out [16-column
      // chunk][4-column piece][row][4] so that one store or load of a warp
      // covers 512 contiguous bytes.
      auto slot_ptr = [&](int sl) {
        return p.sk_part + (int64_t)(sl * 2 + (int)rank) * (GBM * 256) + ltid * 4;
      };
      if (whole) {
        for (int col = 0; col < BN && ok; col += 16) {
          uint32_t v[16];
          tmem_ld16(tbase + col, v);
          tmem_ld_wait();
          float a[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) a[j] = __uint_as_float(v[j]);
          if (c0 + col < p.out_cols) store_out(c0 + col, a);
        }
      } else if (ok) {
        // Part of a tile: store this segment's fp32 sums in the cluster's
        // slot (first segment 2c, last 2c + 1), count it in, and let the
        // last of the tile's clusters add the slots in cluster order.
        float *mine = slot_ptr(2 * sc.c + (sg.t == first_tile ? 0 : 1));
        for (int col = 0; col < BN; col += 16) {
          uint32_t v[16];
          tmem_ld16(tbase + col, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 4; ++j)
            __stcg(reinterpret_cast<float4 *>(mine + ((col >> 2) + j) * (GBM * 4)),
                   make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                               __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3])));
        }
      }
      // This warp is done reading accumulator b: free it for the segment after next.
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader)
          mbar_arrive(acc_empty(b));
        else
          mbar_arrive_remote(mapa_shared(acc_empty(b), 0));
      }
      // The named barriers below involve all 4 epilogue warps whatever their
      // wait returned (a warp whose wait timed out still takes part).
      if (!whole) {
        const int c_first = sc.owner(sg.t * num_k);
        const int c_last = sc.owner(sg.t * num_k + num_k - 1);
        __threadfence();
        named_bar_sync(1, 128);
        if (ltid == 0) {
          int *cnt = p.sk_count + 2 * c_last + (int)rank;
          const int prev = atomicAdd(cnt, 1);
          const bool last = prev == c_last - c_first;
          if (last) atomicExch(cnt, 0);  // every contributor has counted in
          *last_flag = last ? 1 : 0;
        }
        named_bar_sync(1, 128);
        const bool last = *last_flag != 0;
        named_bar_sync(1, 128);  // the flag is read before the next segment rewrites it
        if (last && ok) {
          __threadfence();
          for (int col = 0; col < BN && c0 + col < p.out_cols; col += 16) {
            float a[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) a[j] = 0.f;
            for (int cc = c_first; cc <= c_last; ++cc) {
              const float *src = slot_ptr(2 * cc + (sg.t == sc.ubeg(cc) / num_k ? 0 : 1));
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const float4 w = __ldcg(reinterpret_cast<const float4 *>(
                    src + ((col >> 2) + j) * (GBM * 4)));
                a[4 * j] += w.x;
                a[4 * j + 1] += w.y;
                a[4 * j + 2] += w.z;
                a[4 * j + 3] += w.w;
              }
            }
            store_out(c0 + col, a);
          }
        }
      }
    }
  } else if (warp == kTmaWarp) {
    // --------------------------------------------------------- TMA producer
    if (lane == 0) {
      const int ncb = RP / 16;
      // LoRA operand halves of the segment (segment index j, tile t) into
      // buffer j & 1; only the segment that starts a tile uses them.
      auto issue_up = [&](int j, const Seg &sg) {
        const int b = j & 1;
        if (!mbar_wait_bounded(up_empty(b), ((uint32_t)(j >> 1) & 1u) ^ 1u, cta_err, p.status))
          return false;
        if (sg.kb0 != 0) {
          mbar_arrive(up_full(b));
          return true;
        }
        int mt, nt;
        sc.coords(sg.t, mt, nt);
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
      int it = 0;
      Seg nxt = seg_at(sc, sc.u0);
      if (sc.u0 < sc.u1) {
        ok = issue_up(0, nxt);
        up_issued += ok;
      }
      for (int u = sc.u0; u < sc.u1 && ok; ++it) {
        const Seg sg = nxt;
        u = sg.t * num_k + sg.kb1;
        if (u < sc.u1) {  // next segment's LoRA operands, one segment ahead
          nxt = seg_at(sc, u);
          ok = issue_up(it + 1, nxt);
          up_issued += ok;
        }
        int mt, nt;
        sc.coords(sg.t, mt, nt);
        const int m0 = mt * (2 * GBM) + (int)rank * GBM;
        for (int kb = sg.kb0; kb < sg.kb1 && ok; ++kb) {
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
    // The whole warp runs the loop in step (waits agreed with __all_sync);
    // one elected lane issues each MMA and commit.
    const uint32_t idesc_main = make_idesc_bf16(2 * GBM, BN, kDx);
    const uint32_t idesc_up = make_idesc_bf16(2 * GBM, BN, false);
    // Descriptors of stage 0, k step 0.  A stage offset (SB bytes) and the
    // k steps add to the 14-bit start-address field (addresses stay below
    // 256 KB, so no carry leaves it).
    const uint64_t a_desc0 = make_sdesc(smem0, 16, 1024, kSwz128);
    const uint64_t b_desc0 = kDx ? make_sdesc(smem0 + kABytes, 8192, 1024, kSwz128)
                                 : make_sdesc(smem0 + kABytes, 16, 1024, kSwz128);
    constexpr uint32_t kBStep = kDx ? (2048u >> 4) : (32u >> 4);
    const uint32_t sstep = (uint32_t)SB >> 4;
    uint32_t soff = 0;
    int stage = 0;
    uint32_t ph = 0;
    bool ok = true;
    int last_acc = -1;
    int it = 0;
    for (int u = sc.u0; u < sc.u1 && ok; ++it) {
      const Seg sg = seg_at(sc, u);
      u = sg.t * num_k + sg.kb1;
      const int b = it & 1;
      const uint32_t use_ph = (uint32_t)(it >> 1) & 1u;
      ok = mbar_wait_bounded(acc_empty(b), use_ph ^ 1u, cta_err, p.status);
      if (ok) ok = mbar_wait_bounded(up_full(b), use_ph, cta_err, p.status);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t d = tmem + (uint32_t)(b * kAccCols);
      // LoRA term first, once per tile: D = (s.t) . B^T  (or (s.u) . A for dX)
      const bool lora = sg.kb0 == 0;
      if (lora) {
        for (int cb = 0; cb < RP / 16; ++cb) {
          const uint64_t ad = make_sdesc(upa_u + b * UPA + cb * (GBM * 32), 16, 256, kSwz32);
          const uint64_t bd = make_sdesc(upb_u + b * UPB + cb * (kHalfN * 32), 16, 256, kSwz32);
          tc_mma2_elect(d, ad, bd, idesc_up, cb > 0 ? 1u : 0u);
        }
      }
      tc_commit2_mc_elect(up_empty(b), 0x3);
      uint32_t acc0 = lora ? 1u : 0u;  // the first base MMA of a tile's later segment starts D
      for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(full_bar(stage), ph, cta_err, p.status));
        if (!ok) break;
        tc_fence_after();
        const uint64_t ad = a_desc0 + soff, bd = b_desc0 + soff;
        tc_mma2_elect(d, ad, bd, idesc_main, acc0);
        acc0 = 1u;
#pragma unroll
        for (int kk = 1; kk < 4; ++kk)
          tc_mma2_elect(d, ad + 2u * kk, bd + kBStep * kk, idesc_main, 1u);
        tc_commit2_mc_elect(empty_bar(stage), 0x3);
        if (++stage == S) {
          stage = 0;
          ph ^= 1;
          soff = 0;
        } else {
          soff += sstep;
        }
      }
      tc_commit2_mc_elect(acc_full(b), 0x3);
      last_acc = it;
    }
    // Error path: every issued MMA retired before TMEM is freed.
    if (lane == 0 && ld_shared_volatile(cta_err) && last_acc >= 0)
      mbar_drain(acc_full(last_acc & 1), (uint32_t)(last_acc >> 1) & 1u);
    __syncwarp();
  } else {
    // ----------------------------------------------- relay (peer CTA)
    // Forwards, per segment, "this CTA's LoRA operand halves landed" and
    // then, per stage, "this CTA's half of stage s is ready" (its TMA bytes
    // landed and the 4 warps of the producer group arrived) to the leader's
    // barriers, in the order the leader consumes them.
    if (lane == 0) {
      // The leader's barrier array, as seen from this CTA.
      const uint32_t lead_bars = mapa_shared(smem_u32(bars), 0);
      int stage = 0;
      uint32_t ph = 0;
      bool ok = true;
      int it = 0;
      for (int u = sc.u0; u < sc.u1 && ok; ++it) {
        const Seg sg = seg_at(sc, u);
        u = sg.t * num_k + sg.kb1;
        const int b = it & 1;
        ok = mbar_wait_bounded(up_full(b), (uint32_t)(it >> 1) & 1u, cta_err, p.status);
        if (!ok) break;
        mbar_arrive_remote(lead_bars + 8u * (uint32_t)(2 * S + b));
        for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
          ok = mbar_wait_bounded(full_bar(stage), ph, cta_err, p.status);
          if (!ok) break;
          mbar_arrive_remote(lead_bars + 8u * (uint32_t)stage);
          if (++stage == S) {
            stage = 0;
            ph ^= 1;
          }
        }
      }
    }
    __syncwarp();
  }

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the pair is done with TMEM and with each other's smem
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc2(tmem, 2 * kAccCols);
  }
}

// ------------------------------------------------------------ host launcher
namespace {
// Clusters of the kernel that fit on the current device at once, cached per
// (kernel, shared-memory size, device).
cudaError_t max_active_clusters(bool dx, int smem, int *out) {
  static bool attr_set[2] = {false, false};
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
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if (cached_smem[dx] != smem || cached_dev[dx] != dev) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kGemmThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attrs[1];
    attrs[0].id = cudaLaunchAttributeClusterDimension;
    attrs[0].val.clusterDim.x = 2;
    attrs[0].val.clusterDim.y = 1;
    attrs[0].val.clusterDim.z = 1;
    cfg.attrs = attrs;
    cfg.numAttrs = 1;
    int n = 0;
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
  *out = cached_clusters[dx];
  return cudaSuccess;
}

// Pair-tile width for whole-tile launches: the candidate minimising (waves
// of tiles over the clusters) x (tile width + 1100).  A contraction step of
// a pair tile costs about 0.33 us + 0.29 ns per column on B300 (the MMA
// issue, not the tensor math, sets the pace of narrow tiles), i.e. a fixed
// part worth ~1100 columns.  The dX operand is MN-major in 64-column atoms
// per CTA, so there only 128 or 256.
int pick_bn(int M, int out_cols, bool dx, int clusters) {
  static const int fwd_c[] = {256, 224, 192, 160, 128};
  static const int dx_c[] = {256, 128};
  const int *c = dx ? dx_c : fwd_c;
  const int nc = dx ? 2 : 5;
  const int mp = (M + 2 * GBM - 1) / (2 * GBM);
  int best = 256;
  long best_cost = -1;
  for (int i = 0; i < nc; ++i) {
    const long tiles = (long)mp * ((out_cols + c[i] - 1) / c[i]);
    const long waves = (tiles + clusters - 1) / clusters;
    const long cost = waves * (c[i] + 1100);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = c[i];
    }
  }
  return best;
}
}  // namespace

int gemm_cluster_bound() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 2)
    return 74;
  return n / 2;
}

// Whole tiles (width from pick_bn) unless they would keep fewer than half of
// the clusters' wave slots busy; then, given a split-tile area, split tiles
// with an equal share of units per cluster, as long as a share is at least 8
// contraction blocks.  (A split tile costs its last cluster a pass over the
// fp32 partials at the end of its range, so splitting only pays when most
// clusters would otherwise idle.)
cudaError_t gemm_plan(bool dx, int M, int out_cols, int kdim, int r_pad, int sk_slots_clusters,
                      GemmPlan *plan) {
  int maxc = 0;
  cudaError_t e = max_active_clusters(dx, gemm_smem_bytes(gemm_pick_stages(r_pad), r_pad), &maxc);
  if (e != cudaSuccess) return e;
  const int64_t mp = (M + 2 * GBM - 1) / (2 * GBM);
  const int64_t num_k = (kdim + GBK - 1) / GBK;
  auto tiles_of = [&](int bn) { return mp * ((out_cols + bn - 1) / bn); };
  if ((int64_t)tiles_of(128) * num_k >= ((int64_t)1 << 31)) return cudaErrorInvalidValue;
  const int bn = pick_bn(M, out_cols, dx, maxc);
  const int64_t T = tiles_of(bn);
  const int64_t waves = (T + maxc - 1) / maxc;
  const bool busy = T * 2 >= waves * maxc;
  const int64_t U = tiles_of(GBN) * num_k;
  const int skc = sk_slots_clusters < maxc ? sk_slots_clusters : maxc;
  if (!busy && skc > 0 && U / skc >= 8) {
    plan->bn = GBN;
    plan->sk = 1;
    plan->clusters = skc;
    return cudaSuccess;
  }
  plan->bn = bn;
  plan->sk = 0;
  plan->clusters = (int)(T < maxc ? T : maxc);
  return cudaSuccess;
}

cudaError_t launch_gemm(bool dx, const CUtensorMap &tmA, const CUtensorMap &tmL1,
                        const CUtensorMap &tmL2, const GemmArgs &args, cudaStream_t s) {
  if (args.clusters < 1) return cudaSuccess;  // nothing to compute
  if (args.sk && (!args.sk_part || !args.sk_count || args.clusters > args.sk_slots_clusters))
    return cudaErrorInvalidValue;
  const int smem = gemm_smem_bytes(args.stages, args.r_pad);
  int maxc = 0;
  cudaError_t e = max_active_clusters(dx, smem, &maxc);
  if (e != cudaSuccess) return e;
  if (args.clusters > maxc) return cudaErrorInvalidValue;  // all clusters must be resident
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * args.clusters, 1, 1);
  cfg.blockDim = dim3(kGemmThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = 2;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  attrs[1] = pdl_attr();
  cfg.attrs = attrs;
  cfg.numAttrs = 2;
  if (dx)
    e = cudaLaunchKernelEx(&cfg, qlora_gemm_kernel<true>, tmA, tmL1, tmL2, args);
  else
    e = cudaLaunchKernelEx(&cfg, qlora_gemm_kernel<false>, tmA, tmL1, tmL2, args);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

int gemm_pick_stages(int r_pad) {
  for (int st = 7; st >= 2; --st)
    if (gemm_smem_bytes(st, r_pad) <= 232448) return st;
  return 0;
}

}  // namespace qlora
