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
//   - Every warp owns whole 32-row pairs of tiles over the CTA's K slice and
//     keeps their partial sums in registers: the main loop has no block-wide
//     synchronisation.  A three-slot register ring prefetches the packed
//     bytes and block constants of the next blocks.
//   - Per 64-weight block the block constant a_hat is factored out:
//       sum_{k in block} w_hat x = a_hat . sum_{k in block} c_idx(k) x_k,
//     and the inner sum runs on the tensor cores (mma.sync m16n8k16, f16
//     operands, f32 accumulation): the 4-bit indices become f16 codepoint
//     pairs through a 256-entry byte table in shared memory, replicated per
//     lane so that 32 random bytes never collide on a bank.
//   - One warp also computes the CTA's slice of t = x A^T on the same x
//     fragments.  The S partial sums meet once, in CTA 0 of the cluster, in
//     rank order (deterministic, no workspace, no atomics), which adds the
//     LoRA term s . t . B^T and writes y.
// The codepoints enter as f16 (error <= 2^-12 relative) and the product
// with a_hat stays in fp32, so the result is within the documented
// tolerance of x . W_hat^T with the bf16-rounded W_hat.
#include "common.cuh"
#include "kernels.h"

namespace qlora {

__constant__ float kNf4Const[16] = {QLORA_NF4_VALUES};

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

// bf16 pair -> f16 pair (both halves), round to nearest.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  return pack_f16x2(bf16_lo(w), bf16_hi(w));
}

// Shared-memory layout of the GEMV kernel (bytes).
struct GemvSmem {
  int tab, xs, part, tpart, tfull, bsm, amax, total;
};
__host__ __device__ inline GemvSmem gemv_smem_layout(int nblk, int MT, int rows_max, int G) {
  GemvSmem L;
  L.tab = 0;  // 32 KB slack, then the 256 x 32 lanes x u32 table at a 32 KB-aligned address
  L.xs = 65536;                                         // nblk x MT x 72 f16
  L.part = L.xs + nblk * MT * kXRowHalves * 2;          // G x rows_max x 16 f32: partial y
  L.tpart = L.part + G * rows_max * 16 * 4;             // 64 j x 16 tok f32: partial t
  L.tfull = L.tpart + 64 * 16 * 4;                      // 16 tok x 64 j f32 (rank 0)
  L.bsm = L.tfull + 16 * 64 * 4;                        // rows_max x 64 bf16 (rank 0)
  L.amax = L.bsm + rows_max * 64 * 2;                   // 16 ints: per-token max |x| bits
  L.total = L.amax + 16 * 4;
  return L;
}

// Packed bytes and block constants of rows (g, g+8) of the two row tiles of
// one 32-row pair, one 64-block.  Raw until use (see the GEMM producer).
struct GemvStep {
  uint2 pk[2][2];
  int code[2][2];
  float cv[2][2];
  uint32_t valid;  // bit (rt * 2 + h)
};

template <int NT>
__global__ void __launch_bounds__(kGemvWarps * 32, 1) qlora_gemv_kernel(const GemvArgs p) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int MT = NT * 8;
  const int nblk = p.slice >> 6;
  const GemvSmem SL = gemv_smem_layout(nblk, MT, p.rows_max, p.kparts);
  const uint32_t tab_u = (smem_u32(smem) + 0x7fffu) & ~0x7fffu;  // 32 KB aligned
  uint16_t *xs = reinterpret_cast<uint16_t *>(smem + SL.xs);
  float *part = reinterpret_cast<float *>(smem + SL.part);
  float *tpart = reinterpret_cast<float *>(smem + SL.tpart);
  float *tfull = reinterpret_cast<float *>(smem + SL.tfull);
  uint16_t *bsm = reinterpret_cast<uint16_t *>(smem + SL.bsm);
  int *amax_bits = reinterpret_cast<int *>(smem + SL.amax);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tq = lane & 3;
  const uint32_t rank = cluster_ctarank();
  const int S = gridDim.y;
  const int RP = (p.r + 15) & ~15;
  const int kc0 = (int)rank * p.slice;
  const int kb0 = kc0 >> 6;
  const int64_t kbr = p.K >> 6;
  const int rp_begin = (int)((int64_t)p.row_pairs * blockIdx.x / p.clusters);
  const int rp_end = (int)((int64_t)p.row_pairs * (blockIdx.x + 1) / p.clusters);
  const int row_lo = rp_begin * 32;
  const int row_hi = min(rp_end * 32, p.N);

  // ---- prologue: codepoint-pair table, B rows (rank 0), x slice as f16
  for (int i = threadIdx.x; i < 256 * 32; i += blockDim.x) {
    const int b = i >> 5;  // uniform across a warp
    const uint32_t v = pack_f16x2(kNf4Const[b >> 4], kNf4Const[b & 15]);
    asm volatile("st.shared.u32 [%0], %1;" ::"r"(tab_u + i * 4), "r"(v) : "memory");
  }
  if (threadIdx.x < 16) amax_bits[threadIdx.x] = 0;
  if (rank == 0) {
    const int per_row = p.r >> 3;
    const int npieces = (row_hi - row_lo) * per_row;
    for (int i0 = threadIdx.x; i0 < npieces; i0 += 4 * blockDim.x) {
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + u * blockDim.x;
        const int ic = i < npieces ? i : 0;
        v[u] = ldg_nc_v4(p.B + (int64_t)(row_lo + ic / per_row) * p.r + (ic % per_row) * 8);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + u * blockDim.x;
        if (i < npieces)
          *reinterpret_cast<uint4 *>(bsm + (i / per_row) * 64 + (i % per_row) * 8) = v[u];
      }
    }
  }
  __syncthreads();
  // x slice: MT tokens x nblk*64 columns, 8 columns per piece.
  const int xpieces = MT * nblk * 8;
  constexpr int kMaxXp = (16 * (kGemvMaxSlice / 8)) / (kGemvWarps * 32);  // 8
  uint4 xv[kMaxXp];
#pragma unroll
  for (int u = 0; u < kMaxXp; ++u) {
    const int i = threadIdx.x + u * blockDim.x;
    const int tok = i / (nblk * 8), col = (i % (nblk * 8)) * 8 + kc0;
    xv[u] = make_uint4(0, 0, 0, 0);
    if (i < xpieces && tok < p.M && col < p.K) xv[u] = ldg_nc_v4(p.x + (int64_t)tok * p.K + col);
  }
#pragma unroll
  for (int u = 0; u < kMaxXp; ++u) {
    const int i = threadIdx.x + u * blockDim.x;
    if (i < xpieces) {
      const uint32_t w[4] = {xv[u].x, xv[u].y, xv[u].z, xv[u].w};
      float m = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) m = fmaxf(m, fmaxf(fabsf(bf16_lo(w[e])), fabsf(bf16_hi(w[e]))));
      atomicMax(&amax_bits[i / (nblk * 8)], __float_as_int(m));
    }
  }
  __syncthreads();
#pragma unroll
  for (int u = 0; u < kMaxXp; ++u) {
    const int i = threadIdx.x + u * blockDim.x;
    if (i < xpieces) {
      const int tok = i / (nblk * 8), c8 = i % (nblk * 8);
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

  // ---- t = x A^T over this CTA's slice (the last warp, before its rows)
  if (warp == kGemvWarps - 1) {
    for (int jt = 0; jt < RP / 16; ++jt) {
      float d[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) d[nt][0] = d[nt][1] = d[nt][2] = d[nt][3] = 0.f;
      for (int blk = 0; blk < nblk; ++blk) {
        const int col = kc0 + blk * 64 + tq * 16;
        uint32_t a0w[8] = {0, 0, 0, 0, 0, 0, 0, 0}, a8w[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int j = jt * 16 + g + 8 * h;
          if (j < p.r && col < p.K) {
            const uint4 u0 = ldg_nc_v4(p.A + (int64_t)j * p.K + col);
            const uint4 u1 = ldg_nc_v4(p.A + (int64_t)j * p.K + col + 8);
            uint32_t *dst = h ? a8w : a0w;
            dst[0] = u0.x, dst[1] = u0.y, dst[2] = u0.z, dst[3] = u0.w;
            dst[4] = u1.x, dst[5] = u1.y, dst[6] = u1.z, dst[7] = u1.w;
          }
        }
        uint32_t xf[4][NT][2];
        load_xf(blk, xf);
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const uint32_t a[4] = {bf16x2_to_f16x2(a0w[2 * jj]), bf16x2_to_f16x2(a8w[2 * jj]),
                                 bf16x2_to_f16x2(a0w[2 * jj + 1]), bf16x2_to_f16x2(a8w[2 * jj + 1])};
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma_f16_16816(d[nt], a, xf[jj][nt][0], xf[jj][nt][1]);
        }
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int tok = nt * 8 + 2 * tq;
        tpart[(jt * 16 + g) * 16 + tok] = d[nt][0] * csc[nt][0];
        tpart[(jt * 16 + g) * 16 + tok + 1] = d[nt][1] * csc[nt][1];
        tpart[(jt * 16 + g + 8) * 16 + tok] = d[nt][2] * csc[nt][0];
        tpart[(jt * 16 + g + 8) * 16 + tok + 1] = d[nt][3] * csc[nt][1];
      }
    }
  }

  // ---- main loop.  A task is (row pair, k part): the CTA's K slice is cut
  // into G = p.kparts parts so that P row pairs x G parts keep all warps
  // busy; task t = rp_local * G + part, warp w runs tasks w, w + 16, ...
  // Step = one 64-block of a task.
  const uint32_t lanebase = tab_u | (lane * 4);
  const int G = p.kparts;
  const int bpp = (nblk + G - 1) / G;  // blocks per part
  const int ntask = (rp_end - rp_begin) * G;
  const int my_tasks = (ntask - warp + kGemvWarps - 1) / kGemvWarps;
  const int steps = my_tasks > 0 ? my_tasks * bpp : 0;
  // Position of a step (task, block within the task), advanced by adds
  // (no runtime divisions in the loop).
  struct Cursor {
    int task, bi;  // task index, block index within the task's part
  };
  auto advance = [&](Cursor &c) {
    if (++c.bi == bpp) {
      c.bi = 0;
      c.task += kGemvWarps;
    }
  };
  auto load_step = [&](const Cursor &c, GemvStep &P) {
    const bool in = c.task < ntask;
    const int rpl = in ? c.task / G : 0;  // once per block, G is small
    const int blk = in ? (c.task - rpl * G) * bpp + c.bi : 0;
    const int rp = rp_begin + rpl;
    const int kb = kb0 + blk;
    const bool kok = in && blk < nblk && kb < kbr;
    P.valid = 0;
#pragma unroll
    for (int rt = 0; rt < 2; ++rt)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int row = rp * 32 + rt * 16 + 8 * h + g;
        const bool ok = kok && row < p.N;
        const int64_t b = ok ? (int64_t)row * kbr + kb : 0;
        P.pk[rt][h] = ldg_nc_v2(p.packed + (ok ? (b << 5) + tq * 8 : 0));
        P.code[rt][h] = ldg_nc_s8(p.codes + (p.use_code ? b : 0));
        P.cv[rt][h] = ldg_nc_f32(p.cvec + (b >> p.cshift));
        P.valid |= ok ? (1u << (rt * 2 + h)) : 0u;
      }
  };
  float acc[2][NT][4];
  auto zero_acc = [&]() {
#pragma unroll
    for (int rt = 0; rt < 2; ++rt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) acc[rt][nt][0] = acc[rt][nt][1] = acc[rt][nt][2] = acc[rt][nt][3] = 0.f;
  };
  auto compute_step = [&](const Cursor &c, const GemvStep &P) {
    const int rpl = c.task / G;
    const int part_i = c.task - rpl * G;
    const int blk = min(part_i * bpp + c.bi, nblk - 1);
    uint32_t xf[4][NT][2];
    load_xf(blk, xf);
#pragma unroll
    for (int rt = 0; rt < 2; ++rt) {
      float tmp[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) tmp[nt][0] = tmp[nt][1] = tmp[nt][2] = tmp[nt][3] = 0.f;
      const uint32_t w0[2] = {P.pk[rt][0].x, P.pk[rt][0].y};
      const uint32_t w8[2] = {P.pk[rt][1].x, P.pk[rt][1].y};
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
        for (int nt = 0; nt < NT; ++nt) mma_f16_16816(tmp[nt], a, xf[j][nt][0], xf[j][nt][1]);
      }
      const float ah0 = ((P.valid >> (rt * 2)) & 1u)
                            ? (p.use_code ? __fmul_rn((float)P.code[rt][0], P.cv[rt][0]) : P.cv[rt][0])
                            : 0.f;
      const float ah8 = ((P.valid >> (rt * 2 + 1)) & 1u)
                            ? (p.use_code ? __fmul_rn((float)P.code[rt][1], P.cv[rt][1]) : P.cv[rt][1])
                            : 0.f;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        acc[rt][nt][0] = fmaf(ah0, tmp[nt][0], acc[rt][nt][0]);
        acc[rt][nt][1] = fmaf(ah0, tmp[nt][1], acc[rt][nt][1]);
        acc[rt][nt][2] = fmaf(ah8, tmp[nt][2], acc[rt][nt][2]);
        acc[rt][nt][3] = fmaf(ah8, tmp[nt][3], acc[rt][nt][3]);
      }
    }
    if (c.bi == bpp - 1) {  // end of a task: scale by 2^e and park in its smem slab
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
      zero_acc();
    }
  };
  zero_acc();
  GemvStep P[3];
  Cursor cc = {warp, 0}, cl = {warp, 0};  // compute / load positions
  load_step(cl, P[0]);
  advance(cl);
  load_step(cl, P[1]);
  advance(cl);
  for (int st0 = 0; st0 < steps; st0 += 3) {
#pragma unroll
    for (int u = 0; u < 3; ++u) {
      if (st0 + u < steps) {
        load_step(cl, P[(u + 2) % 3]);
        advance(cl);
        compute_step(cc, P[u]);
        advance(cc);
      }
    }
  }

  // ---- the G k-part slabs of each row meet in slab 0 (fixed order)
  __syncthreads();
  if (G > 1) {
    const int nrows_l = (rp_end - rp_begin) * 32;
    for (int i = threadIdx.x; i < nrows_l * 16; i += blockDim.x) {
      float v = part[i];
      for (int q = 1; q < G; ++q) v += part[q * p.rows_max * 16 + i];
      part[i] = v;
    }
  }
  // ---- cluster reduction in CTA 0: t first, then y (+ LoRA), rank order
  __syncthreads();
  cluster_sync_all();
  if (rank == 0) {
    for (int i = threadIdx.x; i < 16 * RP; i += blockDim.x) {
      const int tok = i / RP, j = i % RP;
      float v = 0.f;
      for (int q = 0; q < S; ++q) v += ld_dsmem_f32(tpart + j * 16 + tok, (uint32_t)q);
      tfull[tok * 64 + j] = v;
      if (p.t_save && blockIdx.x == 0 && tok < p.M && j < p.r) p.t_save[tok * p.r + j] = v;
    }
    __syncthreads();
    const int nrows = row_hi - row_lo;
    const int nout = nrows * p.M;
    for (int i0 = threadIdx.x; i0 < nout; i0 += 4 * blockDim.x) {
      float v[4] = {0.f, 0.f, 0.f, 0.f};
      for (int q = 0; q < S; ++q) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = i0 + u * blockDim.x;
          const int ic = i < nout ? i : 0;
          v[u] += ld_dsmem_f32(part + (ic % nrows) * 16 + ic / nrows, (uint32_t)q);
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + u * blockDim.x;
        if (i >= nout) continue;
        const int tok = i / nrows, row = i % nrows;
        float l = 0.f;  // LoRA term s . t . B^T
        for (int j = 0; j < p.r; ++j)
          l = fmaf(tfull[tok * 64 + j], __uint_as_float((uint32_t)bsm[row * 64 + j] << 16), l);
        const float y = fmaf(p.s, l, v[u]);
        const int n = row_lo + row;
        if (p.y_bf16)
          reinterpret_cast<__nv_bfloat16 *>(p.y)[(int64_t)tok * p.N + n] = __float2bfloat16_rn(y);
        else
          reinterpret_cast<float *>(p.y)[(int64_t)tok * p.N + n] = y;
      }
    }
  }
  cluster_sync_all();  // keep every CTA's shared memory alive until rank 0 has read it
}

// ------------------------------------------------------------ launchers
// Cluster size S = ceil(K / 2048): the x slice of a CTA fits shared memory.
// (Larger clusters would leave SMs idle: a cluster must fit in one GPC.)
int gemv_plan(int K, int M, int *warps, int *S) {
  if (M < 1 || M > 16) return -1;
  int smin = (K + kGemvMaxSlice - 1) / kGemvMaxSlice;
  if (smin < 1) smin = 1;
  if (smin > 8) return -1;
  *warps = kGemvWarps;
  *S = smin;
  return 0;
}

cudaError_t launch_gemv(GemvArgs a, int num_sms, cudaStream_t s) {
  int warps, S;
  if (gemv_plan(a.K, a.M, &warps, &S) != 0) return cudaErrorInvalidValue;
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
  const size_t smem = gemv_smem_layout(a.slice / 64, nt * 8, a.rows_max, G).total;
  if (smem > 232448) return cudaErrorInvalidValue;
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
