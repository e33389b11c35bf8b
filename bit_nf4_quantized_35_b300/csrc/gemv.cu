// gemv.cu -- memory-bound split-K QLoRA forward for decode-sized M (<= 16
// tokens), sm_103a.
//
// y[m, n] = sum_k x[m, k] w_hat[n, k] + s . sum_j t[m, j] B[n, j],  t = x A^T
// ("QLoRA and 4bit Quantization | QLoRA 与 4-bit 量化", Step 3 formula).
//
// The packed 4-bit weight is the only large operand (N*K/2 bytes), so the
// kernel is built to stream it from HBM once:
//   - A cluster of S CTAs (S <= 8) owns a contiguous range of 32-row pairs
//     of tiles of W; CTA s of the cluster covers one slice of K (at most
//     2048 wide).  The slice of x is staged once in shared memory as f16
//     MMA fragments, each token scaled by an exact power of two so any bf16
//     magnitude fits f16.
//   - A task is (32-row pair, part of the K slice); warp w runs tasks w,
//     w + 16, ... and keeps a task's partial sums in registers, so the main
//     loop has no block-wide synchronisation.  A four-slot register ring
//     brings the packed bytes of the next blocks from one pointer per row
//     (every load of a ring turn is pointer + immediate).
//   - Per 64-weight block the block constant a_hat is factored out:
//       sum_{k in block} w_hat x = a_hat . sum_{k in block} c_idx(k) x_k,
//     and the inner sum runs on the tensor cores (mma.sync m16n8k16, f16
//     operands, f32 accumulation): the 4-bit indices become f16 codepoint
//     pairs through a 256-entry byte table in shared memory, replicated per
//     lane so that 32 random bytes never collide on a bank.  a_hat of the
//     CTA's rows x blocks is computed once, into shared memory.
//   - t = x A^T over the CTA's slice is computed by the warps that have no
//     main-loop task (in parallel with the others' weight stream), else by
//     all warps before their loop.  After the loop every CTA of the cluster
//     sums t over the ranks and finishes its own share of the cluster's
//     rows: the S partial sums of a row meet in rank order (deterministic,
//     no workspace, no atomics), plus the LoRA term s . t . B^T from B rows
//     staged by cp.async.
//   - The codepoint-pair table is built from immediates before the grid
//     dependency wait (programmatic dependent launch); every global access
//     comes after it.
// The codepoints enter as f16 (error <= 2^-12 relative) and the product
// with a_hat stays in fp32, so the result is within the documented
// tolerance of x . W_hat^T with the bf16-rounded W_hat.
#include "common.cuh"
#include "kernels.h"

namespace qlora {

constexpr int kGemvWarps = 16;
constexpr int kGemvMaxSlice = 2048;  // K columns per CTA
constexpr int kXRowHalves = 72;      // padded f16 row of one token in one 64-block

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Same with a zero accumulator in.
__device__ __forceinline__ void mma_f16_16816_z(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                                uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.f));
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

// Codepoint pair of one packed byte: byte kByte (0..3) of word w.  The
// table starts at a 32 KB-aligned shared address `lanebase & ~0x7fff`; entry
// b of lane l is at + b * 128 + l * 4, and `lanebase` = table | l * 4, so the
// address is one shift and one AND-OR.
template <int kByte>
__device__ __forceinline__ uint32_t lut(uint32_t lanebase, uint32_t w) {
  uint32_t off;
  if constexpr (kByte == 0)
    off = ((w << 7) & 0x7f80u) | lanebase;
  else
    off = ((w >> (8 * kByte - 7)) & 0x7f80u) | lanebase;
  // Not volatile: a pure function of its address (the table is written
  // once, before a block barrier), so the compiler may schedule it freely.
  uint32_t v;
  asm("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(off));
  return v;
}

// Codepoint idx (0..15) as a chain of selects between immediates.
template <int I>
__device__ __forceinline__ float nf4_select(int idx, float acc) {
  constexpr float kv[16] = {QLORA_NF4_VALUES};
  constexpr float v = kv[I];
  acc = idx == I ? v : acc;
  if constexpr (I + 1 < 16)
    return nf4_select<I + 1>(idx, acc);
  else
    return acc;
}

// bf16 pair -> f16 pair (both halves), round to nearest.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  return pack_f16x2(bf16_lo(w), bf16_hi(w));
}

// Bytes per staged row of B (r bf16 plus 16 bytes of padding, so that lanes
// reading consecutive rows spread over the banks).
__host__ __device__ inline int gemv_bpitch(int r) { return r * 2 + 16; }

// Shared-memory layout of the GEMV kernel (bytes).
struct GemvSmem {
  int tab, xs, part, tpw, tpart, tfull, bsm, amax, ah, total;
};
// Pitch (floats) of the block-constant array: one padded row of the CTA's
// rows per 64-block, so that lanes storing consecutive blocks of one row
// land in different banks.
__host__ __device__ inline int gemv_ah_pitch(int rows_max) { return rows_max + 1; }
__host__ __device__ inline GemvSmem gemv_smem_layout(int nblk, int MT, int rows_max, int G, int S,
                                                     int r) {
  GemvSmem L;
  L.tab = 0;  // 32 KB slack, then the 256 x 32 lanes x u32 table at a 32 KB-aligned address
  L.xs = 65536;                                   // nblk x MT x 72 f16
  L.part = L.xs + nblk * MT * kXRowHalves * 2;    // G x rows_max x 16 f32: partial y
  L.tpw = L.part + G * rows_max * 16 * 4;         // 16 warps x 16 j x 16 tok f32: per-warp t
  L.tpart = L.tpw + kGemvWarps * 16 * 16 * 4;     // 64 j x 16 tok f32: t over this CTA's slice
  L.tfull = L.tpart + 64 * 16 * 4;                // 64 j x 16 tok f32: t over the whole K
  L.bsm = L.tfull + 64 * 16 * 4;                  // this CTA's share of rows x B row
  L.amax = L.bsm + ((rows_max + S - 1) / S) * gemv_bpitch(r);  // 16 ints: max |x| bits
  L.ah = L.amax + 16 * 4;  // nblk x pitch f32: a_hat of (block, row) of this CTA's range
  L.total = L.ah + nblk * gemv_ah_pitch(rows_max) * 4;
  return L;
}

template <int NT>
__global__ void __launch_bounds__(kGemvWarps * 32, 1) qlora_gemv_kernel(const GemvArgs p) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int MT = NT * 8;
  const int nblk = p.slice >> 6;
  const int S = gridDim.y;
  const GemvSmem SL = gemv_smem_layout(nblk, MT, p.rows_max, p.kparts, S, p.r);
  const uint32_t tab_u = (smem_u32(smem) + 0x7fffu) & ~0x7fffu;  // 32 KB aligned
  uint16_t *xs = reinterpret_cast<uint16_t *>(smem + SL.xs);
  float *part = reinterpret_cast<float *>(smem + SL.part);
  float *tpw = reinterpret_cast<float *>(smem + SL.tpw);
  float *tpart = reinterpret_cast<float *>(smem + SL.tpart);
  float *tfull = reinterpret_cast<float *>(smem + SL.tfull);
  int *amax_bits = reinterpret_cast<int *>(smem + SL.amax);
  float *ah = reinterpret_cast<float *>(smem + SL.ah);
  const uint32_t bsm_u = smem_u32(smem + SL.bsm);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tq = lane & 3;
  const uint32_t rank = cluster_ctarank();
  const int RP = (p.r + 15) & ~15;
  const int kc0 = (int)rank * p.slice;
  const int kb0 = kc0 >> 6;
  const int64_t kbr = p.K >> 6;
  // (row_pairs * clusters < 2^31 for any N the launcher accepts)
  const int rp_begin = (int)((uint32_t)p.row_pairs * blockIdx.x / (uint32_t)p.clusters);
  const int rp_end = (int)((uint32_t)p.row_pairs * (blockIdx.x + 1) / (uint32_t)p.clusters);
  const int row_lo = rp_begin * 32;
  const int row_hi = min(rp_end * 32, p.N);
  // This CTA's share of the cluster's rows in the final reduction.
  const int share = (row_hi - row_lo + S - 1) / S;
  const int sh_lo = min(row_lo + (int)rank * share, row_hi);
  const int sh_hi = min(sh_lo + share, row_hi);
  const int bpitch = gemv_bpitch(p.r);

  // Main-loop work.  A task is (row pair, k part): the CTA's K slice is cut
  // into G = p.kparts parts so that P row pairs x G parts keep all warps
  // busy; task t = rp_local * G + part, warp w runs tasks w, w + 16, ...
  // Step = one 64-block of a task.
  const int G = p.kparts;
  const int bpp = (nblk + G - 1) / G;  // blocks per part
  const int ntask = (rp_end - rp_begin) * G;

  // ---- 1. work that reads no global memory: with programmatic dependent
  // launch it overlaps the tail of the kernel before this one (which may
  // have written any input, the NF4 buffers included).  Codepoint-pair
  // table, from immediates:
  {
    const float mine = nf4_select<0>(lane & 15, 0.f);  // lane l holds codepoint l & 15
    for (int b = warp; b < 256; b += kGemvWarps) {
      // low half: codepoint of the byte's high nibble, high half: low nibble
      const uint32_t v = pack_f16x2(__shfl_sync(0xffffffffu, mine, b >> 4),
                                    __shfl_sync(0xffffffffu, mine, b & 15));
      asm volatile("st.shared.u32 [%0], %1;" ::"r"(tab_u + (b * 32 + lane) * 4), "r"(v) : "memory");
    }
  }
  if (threadIdx.x < 16) amax_bits[threadIdx.x] = 0;
  // ---- 2. wait for the kernel before this one (no-op without programmatic
  // dependent launch), then read the inputs: B rows of this CTA's row share
  // to shared memory (cp.async, waited for before the final reduction), the
  // x slice, and the block constants.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  {
    const int pieces = p.r >> 3;  // 16-byte pieces per B row
    const int nb = (sh_hi - sh_lo) * pieces;
    for (int i = threadIdx.x; i < nb; i += blockDim.x) {
      const int rl = i / pieces, c = i - rl * pieces;
      cp_async16(bsm_u + rl * bpitch + c * 16, p.B + (int64_t)(sh_lo + rl) * p.r + c * 8, 16);
    }
    cp_async_commit();
  }

  // x slice: MT tokens x nblk*64 columns, 8 columns per piece.
  const int xpieces = MT * nblk * 8;
  constexpr int kMaxXp = NT * 4;  // MT x (2048 / 8) pieces over 512 threads
  const int ppt = nblk * 8;  // pieces per token
  uint4 xv[kMaxXp];
  int xtok[kMaxXp], xc8[kMaxXp];  // (token, piece within the token) of piece u
#pragma unroll
  for (int u = 0; u < kMaxXp; ++u) {
    const int i = threadIdx.x + u * blockDim.x;
    xtok[u] = i / ppt;
    xc8[u] = i - xtok[u] * ppt;
    const int col = xc8[u] * 8 + kc0;
    xv[u] = make_uint4(0, 0, 0, 0);
    if (i < xpieces && xtok[u] < p.M && col < p.K)
      xv[u] = ldg_nc_v4(p.x + (int64_t)xtok[u] * p.K + col);
  }

  // block constants a_hat of the CTA's rows x slice blocks (0 outside W):
  // lane = block, warp + 16 i = row, all loads of a thread in one batch
  const int nrows_l = (rp_end - rp_begin) * 32;
  const int ah_pitch = gemv_ah_pitch(p.rows_max);
  if (lane < nblk) {
    constexpr int kAhBatch = NT == 1 ? 14 : 7;  // rows per load batch (registers)
    const bool kin = kb0 + lane < kbr;
    for (int rl0 = warp; rl0 < nrows_l; rl0 += kGemvWarps * kAhBatch) {
      int code[kAhBatch];
      float cv[kAhBatch];
#pragma unroll
      for (int i = 0; i < kAhBatch; ++i) {
        const int row = row_lo + rl0 + kGemvWarps * i;
        const bool ok = kin && rl0 + kGemvWarps * i < nrows_l && row < p.N;
        const int64_t b = ok ? (int64_t)row * kbr + kb0 + lane : 0;
        code[i] = ldg_nc_s8(p.codes + (p.use_code ? b : 0));
        cv[i] = ok ? ldg_nc_f32(p.cvec + (b >> p.cshift)) : 0.f;
      }
#pragma unroll
      for (int i = 0; i < kAhBatch; ++i) {
        const int rl = rl0 + kGemvWarps * i;
        if (rl < nrows_l)
          ah[lane * ah_pitch + rl] = p.use_code ? __fmul_rn((float)code[i], cv[i]) : cv[i];
      }
    }
  }
  __syncthreads();
  // ---- 3. x as f16 MMA fragments, each token scaled by 2^-e (exact)
  // per-token max |x|: all 32 lanes reduce over the lanes of the same token
  // (|x| bits order like the magnitudes), then one shared-memory atomic per
  // (warp, token)
#pragma unroll
  for (int u = 0; u < kMaxXp; ++u) {
    const int i = threadIdx.x + u * blockDim.x;
    const uint32_t w[4] = {xv[u].x, xv[u].y, xv[u].z, xv[u].w};
    float m = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) m = fmaxf(m, fmaxf(fabsf(bf16_lo(w[e])), fabsf(bf16_hi(w[e]))));
    const int key = i < xpieces ? xtok[u] : -1;
    const unsigned same = __match_any_sync(0xffffffffu, key);
    const unsigned mx = __reduce_max_sync(same, __float_as_uint(m));
    if (key >= 0 && lane == __ffs(same) - 1) atomicMax(&amax_bits[key], (int)mx);
  }
  __syncthreads();
#pragma unroll
  for (int u = 0; u < kMaxXp; ++u) {
    const int i = threadIdx.x + u * blockDim.x;
    if (i < xpieces) {
      const int tok = xtok[u], c8 = xc8[u];
      const int E = ((amax_bits[tok] >> 23) & 0xff) - 127;
      const int e = E >= 15 ? E - 14 : 0;
      const float sc = __uint_as_float((uint32_t)(127 - e) << 23);  // 2^-e
      const uint32_t w[4] = {xv[u].x, xv[u].y, xv[u].z, xv[u].w};
      uint4 o;
      o.x = pack_f16x2(bf16_lo(w[0]) * sc, bf16_hi(w[0]) * sc);
      o.y = pack_f16x2(bf16_lo(w[1]) * sc, bf16_hi(w[1]) * sc);
      o.z = pack_f16x2(bf16_lo(w[2]) * sc, bf16_hi(w[2]) * sc);
      o.w = pack_f16x2(bf16_lo(w[3]) * sc, bf16_hi(w[3]) * sc);
      const int blk = c8 >> 3, c = (c8 & 7) * 8;
      *reinterpret_cast<uint4 *>(xs + (blk * MT + tok) * kXRowHalves + c) = o;
    }
  }
  __syncthreads();
  // 2^e of the two tokens (nt*8 + 2tq, +1) whose accumulator columns this lane holds
  float csc[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int E = ((amax_bits[nt * 8 + 2 * tq + i] >> 23) & 0xff) - 127;
      const int e = E >= 15 ? E - 14 : 0;
      csc[nt][i] = __uint_as_float((uint32_t)(127 + e) << 23);
    }

  // B fragments of block `blk` for token tile nt: words (4j,4j+1), (4j+2,4j+3)
  auto load_xf = [&](int blk, uint32_t (&xf)[4][NT][2]) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const uint16_t *src = xs + (blk * MT + nt * 8 + g) * kXRowHalves + tq * 16;
      const uint4 a = *reinterpret_cast<const uint4 *>(src);
      const uint4 b = *reinterpret_cast<const uint4 *>(src + 8);
      xf[0][nt][0] = a.x, xf[0][nt][1] = a.y, xf[1][nt][0] = a.z, xf[1][nt][1] = a.w;
      xf[2][nt][0] = b.x, xf[2][nt][1] = b.y, xf[3][nt][0] = b.z, xf[3][nt][1] = b.w;
    }
  };

  // ---- 4. t = x A^T over this CTA's slice.  Warps with no main-loop task
  // (a CTA with fewer than 16 tasks) compute it while the others stream W;
  // otherwise all warps do, before their main loop.  Work unit = (16-wide j
  // tile jt, block group grp): the blocks grp, grp + gpj, ... of the slice;
  // unit u = jt + grp * JT goes to t-warp u, u + Tw, ...  Each unit's sum is
  // parked in its own slot and the slots are added in group order after the
  // main loop (fixed order).
  const int JT = RP >> 4;
  const int t_first = ntask < kGemvWarps ? ntask : 0;  // first t-warp
  const int Tw = kGemvWarps - t_first;                 // t-warps
  const int gpj = max(1, Tw / JT);                     // block groups per j tile
  if (warp >= t_first) {
    auto load_a = [&](int jt, int blk, uint4 (&av)[2][2]) {
      const int col = kc0 + blk * 64 + tq * 16;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int j = jt * 16 + g + 8 * h;
        const bool ok = blk < nblk && j < p.r && col < p.K;
        const uint16_t *src = p.A + (ok ? (int64_t)j * p.K + col : 0);
        av[h][0] = ok ? ldg_nc_v4(src) : make_uint4(0, 0, 0, 0);
        av[h][1] = ok ? ldg_nc_v4(src + 8) : make_uint4(0, 0, 0, 0);
      }
    };
    auto mma_a = [&](int blk, const uint4 (&av)[2][2], float (&d)[NT][4]) {
      const uint32_t a0w[8] = {av[0][0].x, av[0][0].y, av[0][0].z, av[0][0].w,
                               av[0][1].x, av[0][1].y, av[0][1].z, av[0][1].w};
      const uint32_t a8w[8] = {av[1][0].x, av[1][0].y, av[1][0].z, av[1][0].w,
                               av[1][1].x, av[1][1].y, av[1][1].z, av[1][1].w};
      uint32_t xf[4][NT][2];
      load_xf(blk, xf);
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const uint32_t a[4] = {bf16x2_to_f16x2(a0w[2 * jj]), bf16x2_to_f16x2(a8w[2 * jj]),
                               bf16x2_to_f16x2(a0w[2 * jj + 1]), bf16x2_to_f16x2(a8w[2 * jj + 1])};
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_f16_16816(d[nt], a, xf[jj][nt][0], xf[jj][nt][1]);
      }
    };
    for (int u = warp - t_first; u < JT * gpj; u += Tw) {
      const int jt = u % JT, grp = u / JT;
      float d[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) d[nt][0] = d[nt][1] = d[nt][2] = d[nt][3] = 0.f;
      // two blocks in flight: load the next while the current one multiplies
      uint4 av0[2][2], av1[2][2];
      load_a(jt, grp, av0);
      for (int blk = grp; blk < nblk; blk += 2 * gpj) {
        load_a(jt, blk + gpj, av1);
        mma_a(blk, av0, d);
        if (blk + gpj < nblk) {
          load_a(jt, blk + 2 * gpj, av0);
          mma_a(blk + gpj, av1, d);
        }
      }
      float *tw = tpw + u * 256;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int tok = nt * 8 + 2 * tq;
        tw[g * 16 + tok] = d[nt][0] * csc[nt][0];
        tw[g * 16 + tok + 1] = d[nt][1] * csc[nt][1];
        tw[(g + 8) * 16 + tok] = d[nt][2] * csc[nt][0];
        tw[(g + 8) * 16 + tok + 1] = d[nt][3] * csc[nt][1];
      }
    }
  }

  // ---- 5. main loop.  A task is (row pair, k part): the CTA's K slice is
  // cut into G = p.kparts parts so that P row pairs x G parts keep all warps
  // busy; task t = rp_local * G + part, warp w runs tasks w, w + 16, ...
  // Step = one 64-block: the packed bytes of rows g + 8q (q = rt * 2 + h)
  // come through a register ring from one pointer per row (a whole ring
  // turn's loads are pointer + immediate); a_hat comes from shared memory.
  const uint32_t lanebase = tab_u | (lane * 4);
  constexpr int kRing = 4;  // ring slots (kRing - 1 blocks in flight)
  for (int task = warp; task < ntask; task += kGemvWarps) {
    const int rpl = task / G;
    const int part_i = task - rpl * G;
    const int blk0 = part_i * bpp;
    // blocks of the task inside the slice and inside K (warp-uniform)
    const int nv = max(0, min(min(bpp, nblk - blk0), (int)kbr - (kb0 + blk0)));
    const int row0 = row_lo + rpl * 32 + g;
    const uint8_t *pr[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int row = row0 + 8 * q;
      const int rr = row < p.N ? row : row_lo;  // a_hat is 0 for rows past N
      pr[q] = p.packed + (size_t)rr * (size_t)(p.K >> 1) + (size_t)(kb0 + blk0) * 32 + tq * 8;
    }
    float acc[2][NT][4];
#pragma unroll
    for (int rt = 0; rt < 2; ++rt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) acc[rt][nt][0] = acc[rt][nt][1] = acc[rt][nt][2] = acc[rt][nt][3] = 0.f;
    uint2 P[kRing][4];
#pragma unroll
    for (int u = 0; u + 1 < kRing; ++u)
      if (u < nv) {
#pragma unroll
        for (int q = 0; q < 4; ++q) P[u][q] = ldg_nc_v2(pr[q] + u * 32);
      }
    const float *ahr = ah + blk0 * ah_pitch + rpl * 32 + g;  // a_hat of (block, row g)
    for (int b0 = 0; b0 < nv; b0 += kRing) {
#pragma unroll
      for (int u = 0; u < kRing; ++u) {
        const int b = b0 + u;
        if (b < nv) {
          if (b + kRing - 1 < nv) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
              P[(u + kRing - 1) % kRing][q] = ldg_nc_v2(pr[q] + (u + kRing - 1) * 32);
          }
          uint32_t xf[4][NT][2];
          load_xf(blk0 + b, xf);
          const float *ahb = ahr + b * ah_pitch;
#pragma unroll
          for (int rt = 0; rt < 2; ++rt) {
            float tmp[NT][4];
            const uint32_t w0[2] = {P[u][rt * 2].x, P[u][rt * 2].y};
            const uint32_t w8[2] = {P[u][rt * 2 + 1].x, P[u][rt * 2 + 1].y};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int wi = j >> 1;
              uint32_t a[4];
              if ((j & 1) == 0) {
                a[0] = lut<0>(lanebase, w0[wi]);
                a[1] = lut<0>(lanebase, w8[wi]);
                a[2] = lut<1>(lanebase, w0[wi]);
                a[3] = lut<1>(lanebase, w8[wi]);
              } else {
                a[0] = lut<2>(lanebase, w0[wi]);
                a[1] = lut<2>(lanebase, w8[wi]);
                a[2] = lut<3>(lanebase, w0[wi]);
                a[3] = lut<3>(lanebase, w8[wi]);
              }
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) {
                if (j == 0)
                  mma_f16_16816_z(tmp[nt], a, xf[j][nt][0], xf[j][nt][1]);
                else
                  mma_f16_16816(tmp[nt], a, xf[j][nt][0], xf[j][nt][1]);
              }
            }
            const float ah0 = ahb[rt * 16], ah8 = ahb[rt * 16 + 8];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              acc[rt][nt][0] = fmaf(ah0, tmp[nt][0], acc[rt][nt][0]);
              acc[rt][nt][1] = fmaf(ah0, tmp[nt][1], acc[rt][nt][1]);
              acc[rt][nt][2] = fmaf(ah8, tmp[nt][2], acc[rt][nt][2]);
              acc[rt][nt][3] = fmaf(ah8, tmp[nt][3], acc[rt][nt][3]);
            }
          }
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) pr[q] += kRing * 32;
    }
    // the task's sum, scaled by 2^e, parked in its k part's slab
#pragma unroll
    for (int rt = 0; rt < 2; ++rt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int tok = nt * 8 + 2 * tq;
        float *r0 = part + (part_i * p.rows_max + rpl * 32 + rt * 16 + g) * 16 + tok;
        *reinterpret_cast<float2 *>(r0) =
            make_float2(acc[rt][nt][0] * csc[nt][0], acc[rt][nt][1] * csc[nt][1]);
        *reinterpret_cast<float2 *>(r0 + 8 * 16) =
            make_float2(acc[rt][nt][2] * csc[nt][0], acc[rt][nt][3] * csc[nt][1]);
      }
  }

  // the next kernel may start its own frozen-buffer work on SMs as they free up
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // ---- 6. within the CTA: the G k-part slabs of each row meet in slab 0,
  // and the per-warp t sums in tpart (fixed orders)
  __syncthreads();
  if (G > 1) {
    const int nrows_l = (rp_end - rp_begin) * 32;
    for (int i = threadIdx.x; i < nrows_l * 16; i += blockDim.x) {
      float v = part[i];
      for (int q = 1; q < G; ++q) v += part[q * p.rows_max * 16 + i];
      part[i] = v;
    }
  }
  {
    for (int i = threadIdx.x; i < RP * 16; i += blockDim.x) {
      const int j = i >> 4, tok = i & 15;
      float v = 0.f;
      if (tok < MT)
        for (int grp = 0; grp < gpj; ++grp) v += tpw[((j >> 4) + grp * JT) * 256 + (j & 15) * 16 + tok];
      tpart[i] = v;
    }
  }
  // ---- 7. across the cluster (rank order): every CTA forms the whole-K t,
  // then finishes its share of the rows, y = sum of the ranks' partials + s t B^T
  __syncthreads();
  cluster_sync_all();
  for (int i = threadIdx.x; i < RP * 16; i += blockDim.x) {
    float v = 0.f;
    for (int q = 0; q < S; ++q) v += ld_dsmem_f32(tpart + i, (uint32_t)q);
    tfull[i] = v;
    const int j = i >> 4, tok = i & 15;
    if (p.t_save && rank == 0 && blockIdx.x == 0 && tok < p.M && j < p.r) p.t_save[tok * p.r + j] = v;
  }
  cp_async_wait<0>();
  __syncthreads();
  {
    const int nsh = sh_hi - sh_lo;
    const int nout = nsh * p.M;
    const int pieces = p.r >> 3;
    for (int i0 = threadIdx.x; i0 < nout; i0 += 4 * blockDim.x) {
      int row[4], tok[4];
      float v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + u * blockDim.x;
        const int ic = i < nout ? i : 0;
        row[u] = ic / p.M;
        tok[u] = ic - row[u] * p.M;
        v[u] = 0.f;
      }
      for (int q = 0; q < S; ++q) {
#pragma unroll
        for (int u = 0; u < 4; ++u)
          v[u] += ld_dsmem_f32(part + (sh_lo - row_lo + row[u]) * 16 + tok[u], (uint32_t)q);
      }
      float l[4] = {0.f, 0.f, 0.f, 0.f};  // LoRA term t . B^T
      for (int c = 0; c < pieces; ++c) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint4 bw = lds_v4(bsm_u + row[u] * bpitch + c * 16);
          const float *tc = tfull + c * 8 * 16 + tok[u];
          l[u] = fmaf(tc[0 * 16], bf16_lo(bw.x), l[u]);
          l[u] = fmaf(tc[1 * 16], bf16_hi(bw.x), l[u]);
          l[u] = fmaf(tc[2 * 16], bf16_lo(bw.y), l[u]);
          l[u] = fmaf(tc[3 * 16], bf16_hi(bw.y), l[u]);
          l[u] = fmaf(tc[4 * 16], bf16_lo(bw.z), l[u]);
          l[u] = fmaf(tc[5 * 16], bf16_hi(bw.z), l[u]);
          l[u] = fmaf(tc[6 * 16], bf16_lo(bw.w), l[u]);
          l[u] = fmaf(tc[7 * 16], bf16_hi(bw.w), l[u]);
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + u * blockDim.x;
        if (i < nout) {
          const float y = fmaf(p.s, l[u], v[u]);
          const int64_t o = (int64_t)tok[u] * p.N + sh_lo + row[u];
          if (p.y_bf16)
            reinterpret_cast<__nv_bfloat16 *>(p.y)[o] = __float2bfloat16_rn(y);
          else
            reinterpret_cast<float *>(p.y)[o] = y;
        }
      }
    }
  }
  cluster_sync_all();  // keep every CTA's shared memory alive until the others have read it
}

// ------------------------------------------------------------ launchers
// Cluster size S = ceil(K / 2048): the x slice of a CTA fits shared memory.
// (Larger clusters would leave SMs idle: a cluster must fit in one GPC.)
// Fills the launcher's fields of `a`; -1 when the shape does not fit the
// kernel (more than 16 tokens, K beyond 8 slices, byte offsets past 32 bits,
// or more shared memory than a CTA may have).
static int gemv_config(GemvArgs &a, int num_sms, int *S_out, size_t *smem_out) {
  if (a.M < 1 || a.M > 16) return -1;
  if ((uint64_t)a.N * (uint64_t)a.K / 2 >= (1ull << 32)) return -1;  // 32-bit byte offsets
  int S = (a.K + kGemvMaxSlice - 1) / kGemvMaxSlice;
  if (S < 1) S = 1;
  if (S > 8) return -1;
  a.slice = ((a.K + S - 1) / S + 63) / 64 * 64;
  a.row_pairs = (a.N + 31) / 32;
  int clusters = num_sms / S;
  if (clusters > a.row_pairs) clusters = a.row_pairs;
  if (clusters < 1) clusters = 1;
  a.clusters = clusters;
  const int pairs_max = (a.row_pairs + clusters - 1) / clusters;
  a.rows_max = pairs_max * 32;
  int G = kGemvWarps / (pairs_max > 0 ? pairs_max : 1);
  if (G < 1) G = 1;
  if (G > a.slice / 64) G = a.slice / 64;
  a.kparts = G;
  const int nt = a.M > 8 ? 2 : 1;
  const size_t smem = gemv_smem_layout(a.slice / 64, nt * 8, a.rows_max, G, S, a.r).total;
  if (smem > 232448) return -1;
  *S_out = S;
  *smem_out = smem;
  return 0;
}

int gemv_plan(int N, int K, int M, int r, int num_sms) {
  GemvArgs a{};
  a.N = N;
  a.K = K;
  a.M = M;
  a.r = r;
  int S;
  size_t smem;
  return gemv_config(a, num_sms, &S, &smem);
}

cudaError_t launch_gemv(GemvArgs a, int num_sms, cudaStream_t s) {
  int S;
  size_t smem;
  if (gemv_config(a, num_sms, &S, &smem) != 0) return cudaErrorInvalidValue;
  const int nt = a.M > 8 ? 2 : 1;
  const int clusters = a.clusters;
  const int warps = kGemvWarps;
  // Dynamic shared memory limit raised to what this launch needs (once per
  // new maximum), cluster sizes above 8 never requested.
  static size_t smem_set[2] = {0, 0};
  cudaError_t e;
  if (smem > smem_set[nt - 1]) {
    if (nt == 2)
      e = cudaFuncSetAttribute(qlora_gemv_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem);
    else
      e = cudaFuncSetAttribute(qlora_gemv_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem);
    if (e != cudaSuccess) return e;
    smem_set[nt - 1] = smem;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(clusters, S, 1);
  cfg.blockDim = dim3(warps * 32, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = 1;
  attrs[0].val.clusterDim.y = S;
  attrs[0].val.clusterDim.z = 1;
  // programmatic dependent launch: the kernel waits (griddepcontrol.wait)
  // before reading x, A or B or writing anything
  attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 2;
  if (nt == 2)
    e = cudaLaunchKernelEx(&cfg, qlora_gemv_kernel<2>, a);
  else
    e = cudaLaunchKernelEx(&cfg, qlora_gemv_kernel<1>, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace qlora
