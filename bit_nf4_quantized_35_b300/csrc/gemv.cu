// gemv.cu -- memory-bound QLoRA forward for decode-sized M (<= 16 tokens),
// sm_103a.
//
// y[m, n] = sum_k x[m, k] w_hat[n, k] + s . sum_j t[m, j] B[n, j],  t = x A^T
// ("QLoRA and 4bit Quantization | QLoRA 与 4-bit 量化", Step 3 formula), with
// w_hat = bf16(c_idx . a_hat) exactly as the dequantiser produces it.
//
// Two kernels, launched back to back with programmatic dependent launch:
//   lora_t_decode_kernel  t = x A^T.  CTA kt covers 256 columns of K; its
//     warps (one per 16 rows of A) run bf16 mma.sync with fp32 accumulation
//     and store a partial t; the last CTA to finish (a counter in the
//     workspace, reset afterwards) adds the partials in CTA order.
//   qlora_gemv_kernel     the base product and the LoRA epilogue.  It streams
//     the packed weights as soon as it starts (everything before the t kernel
//     on the stream has completed by then: the t kernel releases its
//     dependents only after its own grid-dependency wait), and waits for the
//     t kernel only before its epilogue reads t.
//
// The weight stream.  The packed weight [N, K/2 bytes] is cut into units of
// 16 rows x 256 columns (a 2 KB tile: 16 rows x 4 blocks of 64).  A cluster
// of S CTAs owns a contiguous range of 16-row tiles; CTA q of the cluster
// covers the q-th slice of the 256-column chunks of K (S and the split are
// chosen on the host to even out the units per SM).  Inside a CTA the units
// (tile major, chunk minor) are shared out as 16 contiguous ranges, one per
// warp; each warp brings its units into its own ring of 2 KB slots with
// tiled TMA loads (128-byte swizzle, one mbarrier per slot), so up to
// 16 x (2 to 4) units are in flight per SM with no register cost.
//
// The arithmetic of a unit (one warp): mma.sync m16n8k16 bf16, A = 16 weight
// rows, B = up to 8 tokens per n-tile, fp32 accumulation.  The contraction
// order inside a unit is free, so lane group tq owns 64-block tq of the unit
// and MMA j covers positions 4j .. 4j+3 of every lane group's block.  A lane
// therefore dequantises rows g and g+8 of one block (64 + 64 weights) with
// two per-block tables T[i] = bf16(c_i . a_hat) indexed by byte permutes (the
// dequantiser's routine, so the MMA operands are the exact bf16 W_hat), and
// reads the matching x values from shared memory, where x is stored with a
// 16-byte XOR swizzle that keeps every fragment load free of bank conflicts.
// Lanes whose token is past M read a zero row of x.
//
// Reduction (fixed order, deterministic, no atomics): a warp's sum over one
// tile's chunks goes to the CTA's tile sums when the warp covered the whole
// tile, else to one of two partial slots of the warp; the slots of a tile
// are added in warp order.  The S CTAs of a cluster then add their tile sums
// in rank order through distributed shared memory, each finishing its share
// of the cluster's rows with the LoRA term s . t . B^T.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace qlora {

constexpr int kGemvWarps = 16;
constexpr int kGemvDepthMax = 4;     // TMA ring slots per warp (4 down to 2, as shared memory allows)
constexpr int kUnitBytes = 2048;     // 16 rows x 128 packed bytes
constexpr int kChunk = 256;          // columns of K per unit
constexpr int kTWarps = 4;           // t kernel: one warp per 16 rows of A (r <= 64)

// The MMAs are plain register functions (no volatile): the compiler may
// interleave them with the shared-memory loads that feed them.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float ld_dsmem_f32(uint32_t local_addr, uint32_t rank) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(local_addr), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
  return v;
}

__device__ __forceinline__ uint4 ldg_v4_or_zero(const uint16_t *p, bool ok) {
  return ok ? ldg_nc_v4(p) : make_uint4(0, 0, 0, 0);
}

// ------------------------------------------------------------- t = x A^T
// Grid: ceil(K / 256) CTAs of kTWarps warps.  tpart [gridDim.x][M][RP],
// tfin [M][RP] (fp32, workspace), counter: one int, zero between calls.
// With `mask` (LoRA dropout keep bits of x, wpr words per row) the dropped
// elements of x count as zero and t is scaled by keep_scale.
__global__ void __launch_bounds__(kTWarps * 32) lora_t_decode_kernel(
    const uint16_t *__restrict__ x, int M, int K, const uint16_t *__restrict__ A, int r, int RP,
    float *__restrict__ tpart, float *__restrict__ tfin, int *__restrict__ counter,
    float *__restrict__ t_save, const uint32_t *__restrict__ mask, int wpr, float keep_scale) {
  __shared__ int last_s;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tq = lane & 3;
  const int kt = blockIdx.x;
  if (warp * 16 < RP) {
    const int blk = kt * 4 + tq;  // this lane group's 64-block of K
    const bool kin = blk * 64 < K;
    const int j0 = warp * 16 + g, j1 = j0 + 8;
    const uint16_t *a0p = A + (int64_t)(j0 < r ? j0 : 0) * K + (int64_t)(kin ? blk : 0) * 64;
    const uint16_t *a1p = A + (int64_t)(j1 < r ? j1 : 0) * K + (int64_t)(kin ? blk : 0) * 64;
    const bool ok0 = kin && j0 < r, ok1 = kin && j1 < r;
    float d[2][4] = {};
    // every load of the lane first (plain read-only loads the compiler may
    // schedule freely), then the MMAs
    const uint4 z4 = make_uint4(0, 0, 0, 0);
    uint4 ag[8], ah[8], xv[2][8];
    uint32_t kw[2][2];
#pragma unroll
    for (int wi = 0; wi < 8; ++wi) {
      ag[wi] = ok0 ? __ldg(reinterpret_cast<const uint4 *>(a0p + 8 * wi)) : z4;
      ah[wi] = ok1 ? __ldg(reinterpret_cast<const uint4 *>(a1p + 8 * wi)) : z4;
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int tok = nt * 8 + g;
      const bool okx = kin && tok < M;
      const uint16_t *xr = x + (int64_t)(okx ? tok : 0) * K + (int64_t)(kin ? blk : 0) * 64;
#pragma unroll
      for (int wi = 0; wi < 8; ++wi)
        xv[nt][wi] = okx ? __ldg(reinterpret_cast<const uint4 *>(xr + 8 * wi)) : z4;
      // dropout: the block's 64 columns are two keep words
      kw[nt][0] = kw[nt][1] = 0xffffffffu;
      if (mask && okx) {
        kw[nt][0] = __ldg(mask + (int64_t)tok * wpr + blk * 2);
        kw[nt][1] = __ldg(mask + (int64_t)tok * wpr + blk * 2 + 1);
      }
    }
#pragma unroll
    for (int wi = 0; wi < 8; ++wi) {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        uint4 v = xv[nt][wi];
        if (mask) {  // columns blk*64 + 8wi .. +7: byte (wi & 3) of word wi / 4
          uint32_t mk[4];
          keep_masks((kw[nt][wi >> 2] >> (8 * (wi & 3))) & 0xffu, mk);
          v.x &= mk[0], v.y &= mk[1], v.z &= mk[2], v.w &= mk[3];
        }
        mma_bf16(d[nt], ag[wi].x, ah[wi].x, ag[wi].y, ah[wi].y, v.x, v.y);
        mma_bf16(d[nt], ag[wi].z, ah[wi].z, ag[wi].w, ah[wi].w, v.z, v.w);
      }
    }
    float *tp = tpart + (int64_t)kt * M * RP;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int tok = nt * 8 + 2 * tq;
      if (tok < M) {
        tp[tok * RP + j0] = keep_scale * d[nt][0];
        tp[tok * RP + j1] = keep_scale * d[nt][2];
      }
      if (tok + 1 < M) {
        tp[(tok + 1) * RP + j0] = keep_scale * d[nt][1];
        tp[(tok + 1) * RP + j1] = keep_scale * d[nt][3];
      }
    }
  }
  // The last CTA to finish adds the partials in CTA order.
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    last_s = atomicAdd(counter, 1) == (int)gridDim.x - 1;
  }
  __syncthreads();
  if (!last_s) return;
  __threadfence();
  for (int i = threadIdx.x; i < M * RP; i += blockDim.x) {
    float v = 0.f;
    for (int q = 0; q < (int)gridDim.x; ++q) v += __ldcg(tpart + (int64_t)q * M * RP + i);
    tfin[i] = v;
    const int tok = i / RP, j = i - tok * RP;
    if (t_save && j < r) t_save[tok * r + j] = v;
  }
  if (threadIdx.x == 0) *counter = 0;
}

// ------------------------------------------------------------ main kernel
struct GemvSmem {
  int ring, xs, xstride, part, tsum, tfin, bs, wr, bars, err, total;
};
__host__ __device__ inline GemvSmem gemv_smem(int M, int MT, int slice_chunks, int tiles_max,
                                              int RP, int depth, int S) {
  GemvSmem L;
  L.ring = 0;  // 16 warps x depth slots x 2 KB, 1024-byte aligned
  L.xs = L.ring + kGemvWarps * depth * kUnitBytes;
  L.xstride = slice_chunks * kChunk * 2;                 // bytes per token row
  L.part = L.xs + (M + 1) * L.xstride;                   // x rows, then a zero row
  // [16 warps][2][16 rows][MT] f32 partial sums follow
  L.tsum = L.part + kGemvWarps * 2 * 16 * MT * 4;        // [tiles_max][16 rows][MT] f32
  L.tfin = L.tsum + tiles_max * 16 * MT * 4;             // [M][RP] f32
  L.bs = L.tfin + M * RP * 4;                            // B rows of the epilogue share
  L.wr = L.bs + ((tiles_max * 16 + S - 1) / S) * RP * 2;  // warp ranges of the tiles
  L.bars = L.wr + (2 * tiles_max + kGemvWarps) * 4;      // [16][depth] mbarriers
  L.bars = (L.bars + 7) & ~7;
  L.err = L.bars + kGemvWarps * depth * 8;
  L.total = L.err + 16 + 1024;                           // + alignment slack of the base
  return L;
}


// Physical 16-byte slot of logical slot s of token row tok in the x tile: a
// lane's eight fragment loads of one unit, and the loads of the 8 lanes of a
// quarter warp, fall on distinct bank groups.
__device__ __forceinline__ int xswz(int tok, int s) {
  return s ^ (((s >> 3) & 3) | ((tok & 1) << 2));
}

template <int NT>
__global__ void __launch_bounds__(kGemvWarps * 32, 1) qlora_gemv_kernel(
    const __grid_constant__ CUtensorMap tmW, const GemvArgs p) {
  extern __shared__ uint8_t smem_raw[];
  constexpr int MT = NT * 8;
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t *smem = smem_raw + (base - smem_u32(smem_raw));
  const int depth = p.depth;
  const GemvSmem SL = gemv_smem(p.M, MT, p.slice_chunks, p.tiles_max, p.RP, depth, p.S);
  const uint32_t ring_u = base + SL.ring;
  const uint32_t xs_u = base + SL.xs;
  float *part = reinterpret_cast<float *>(smem + SL.part);
  float *tsum = reinterpret_cast<float *>(smem + SL.tsum);
  float *tfin = reinterpret_cast<float *>(smem + SL.tfin);
  const uint32_t bars_u = base + SL.bars;
  const uint32_t err_u = base + SL.err;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tq = lane & 3;
  const int S = p.S;
  const uint32_t rank = cluster_rank();
  const int cl = blockIdx.x / S;
  // tiles of this cluster, chunks (of 256 columns) of this CTA
  const int t0 = (int)((int64_t)p.tiles_total * cl / p.clusters);
  const int t1 = (int)((int64_t)p.tiles_total * (cl + 1) / p.clusters);
  const int Tc = t1 - t0;
  const int Ctot = (p.K + kChunk - 1) / kChunk;
  const int c0 = (int)rank * p.slice_chunks;
  const int Cc = max(0, min(p.slice_chunks, Ctot - c0));
  const int U = Tc * Cc;
  const int u0 = U * warp / kGemvWarps, u1 = U * (warp + 1) / kGemvWarps;
  const int kbr = p.K >> 6;  // 64-chunks per weight row

  if (threadIdx.x < kGemvWarps * depth) mbar_init(bars_u + threadIdx.x * 8, 1);
  if (threadIdx.x == 0) st_shared_volatile(err_u, 0u);
  fence_barrier_init();
  __syncthreads();

  // ---- 1. copies that the weight stream would queue behind go out first:
  // the x slice (tokens < M, zero past K, and a zero row M read by lanes
  // whose token is past M) and the B rows of this CTA's epilogue share
  // (plain async copies; everything before the t kernel on the stream has
  // completed: the t kernel releases its dependents only after its own
  // grid-dependency wait)
  const int spr = p.slice_chunks * (kChunk / 8);  // 16-byte slots per token row
  {
    const int kc0 = c0 * kChunk;
    for (int i = threadIdx.x; i < (p.M + 1) * spr; i += blockDim.x) {
      const int tok = i / spr, s = i - tok * spr;
      const int col = kc0 + s * 8;
      const bool in = tok < p.M && col < p.K;
      cp_async16(xs_u + tok * SL.xstride + xswz(tok, s) * 16,
                 p.x + (in ? (int64_t)tok * p.K + col : 0), in ? 16u : 0u);
    }
    cp_async_commit();
  }
  const int row0 = t0 * 16;
  const int nrows = min(t1 * 16, p.N) - row0;
  const int share = (nrows + S - 1) / S;
  const int r_lo = min((int)rank * share, nrows), r_hi = min(r_lo + share, nrows);
  const int nr = r_hi - r_lo;
  {
    const int pieces = nr * p.r / 8;  // rows are contiguous: r * 2 bytes each, r % 8 == 0
    const uint16_t *src = p.B + (int64_t)(row0 + r_lo) * p.r;
    for (int i = threadIdx.x; i < pieces; i += blockDim.x)
      cp_async16(base + SL.bs + i * 16, src + (int64_t)i * 8, 16u);
    cp_async_commit();
  }

  // ---- 2. the first units of every warp's ring.  Units are walked with
  // (tile, chunk) cursors, chunk fastest.
  auto issue = [&](int tile, int chunk, int slot) {
    const uint32_t bar = bars_u + (warp * depth + slot) * 8;
    mbar_arrive_expect_tx(bar, kUnitBytes);
    tma_load_2d(ring_u + (warp * depth + slot) * kUnitBytes, &tmW, bar,
                (c0 + chunk) * 128, (t0 + tile) * 16);
  };
  const int ut0 = Cc > 0 ? u0 / Cc : 0, uc0 = Cc > 0 ? u0 - ut0 * Cc : 0;  // first unit
  int it_t = ut0, it_c = uc0;  // issue cursor
  auto step = [&](int &t, int &c) {
    if (++c == Cc) {
      c = 0;
      ++t;
    }
  };
  if (lane == 0) {
    tma_prefetch_desc(&tmW);
    for (int i = 0; i < depth && u0 + i < u1; ++i) {
      issue(it_t, it_c, i);
      step(it_t, it_c);
    }
  }

  // ---- 3. the warp ranges of the tiles for the combine step (first and
  // last warp of tile t; first tile of warp w)
  int *wr = reinterpret_cast<int *>(smem + SL.wr);
  if (threadIdx.x < Tc) {
    auto warp_of = [&](int uu) { return (kGemvWarps * (uu + 1) - 1) / U; };
    wr[2 * threadIdx.x] = warp_of(threadIdx.x * Cc);
    wr[2 * threadIdx.x + 1] = warp_of((threadIdx.x + 1) * Cc - 1);
  }
  if (threadIdx.x < kGemvWarps)
    wr[2 * p.tiles_max + threadIdx.x] = Cc > 0 ? (U * (int)threadIdx.x / kGemvWarps) / Cc : 0;
  cp_async_wait<1>();  // this thread's x pieces have landed (the B rows may not have)

  // block constant a_hat of weight row n, 64-chunk kc of that row (0 outside W)
  // (loads clamped into the arrays, the value then zeroed: no branches)
  // (32-bit indices: the plan admits only weights with N * K / 64 < 2^31)
  auto ahat_of = [&](int n, int kc) -> float {
    const bool in = n < p.N && kc < kbr;
    const int b = in ? (n * kbr + kc) >> p.bshift : 0;
    const float cv = ldg_nc_f32(p.cvec + (b >> p.cshift));
    const float a = p.use_code ? __fmul_rn((float)ldg_nc_s8(p.codes + b), cv) : cv;
    return in ? a : 0.f;
  };
  __syncthreads();  // x and the warp ranges staged

  // ---- 4. main loop.  The contraction order inside a unit is free, so lane
  // group tq owns 64-block tq of the unit and MMA j covers positions
  // 4j .. 4j+3 of every lane group's block: a lane dequantises rows g and g+8
  // of one whole block with the block's scaled table (the dequantiser's
  // routine), so the MMA operands are the exact bf16 w_hat.
  const int tok_lo = g, tok_hi = 8 + g;  // this lane's tokens in n-tiles 0 and 1
  float acc[NT][4];
  int cur = -1, seg = 0;
  bool ok = true;
  auto flush = [&](int tile) {
    const bool whole = tile * Cc >= u0 && (tile + 1) * Cc <= u1;
    float *dst = whole ? tsum + tile * 16 * MT : part + (warp * 2 + (seg == 0 ? 0 : 1)) * 16 * MT;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int tok = nt * 8 + 2 * tq;
      dst[g * MT + tok] = acc[nt][0];
      dst[g * MT + tok + 1] = acc[nt][1];
      dst[(g + 8) * MT + tok] = acc[nt][2];
      dst[(g + 8) * MT + tok + 1] = acc[nt][3];
    }
    ++seg;
  };
  // a_hat of the lane's two rows in block tq, loaded one unit ahead
  auto ahat_unit = [&](int tile, int chunk, float &a, float &b) {
    const int kc = (c0 + chunk) * 4 + tq;
    a = ahat_of((t0 + tile) * 16 + g, kc);
    b = ahat_of((t0 + tile) * 16 + g + 8, kc);
  };
  // Shared-memory reads below are ordinary C++ loads (the compiler schedules
  // them; the mbarrier waits and the proxy fence are compiler barriers).
  // x slot of (token, block tq, positions 8 wi .. 8 wi + 7) of chunk c: row
  // tok, slot c * 32 + tq * 8 + (wi ^ x3), x3 = tq | (tok & 1) << 2 (xswz with
  // (s >> 3) & 3 = tq); lanes whose token is past M read the zero row.
  int xoff[8];
#pragma unroll
  for (int wi = 0; wi < 8; ++wi) xoff[wi] = wi ^ (tq | ((g & 1) << 2));
  const bool xv_lo = tok_lo < p.M, xv_hi = tok_hi < p.M;
  const uint4 *xr_lo =
      reinterpret_cast<const uint4 *>(smem + SL.xs + (xv_lo ? tok_lo : p.M) * SL.xstride) + tq * 8;
  const uint4 *xr_hi =
      reinterpret_cast<const uint4 *>(smem + SL.xs + (xv_hi ? tok_hi : p.M) * SL.xstride) + tq * 8;
  float ah_g = 0.f, ah_h = 0.f;
  int tile = ut0, chunk = uc0;  // consume cursor
  if (u0 < u1) ahat_unit(tile, chunk, ah_g, ah_h);
  int done = 0;  // units consumed
  int slot = 0;
  uint32_t phase = 0;
  for (int i = 0; i < u1 - u0; ++i) {
    if (tile != cur) {
      if (cur >= 0) flush(cur);
      cur = tile;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
    }
    int ntile = tile, nchunk = chunk;
    step(ntile, nchunk);
    float nah_g = 0.f, nah_h = 0.f;
    if (i + 1 < u1 - u0) ahat_unit(ntile, nchunk, nah_g, nah_h);
    const uint32_t bar = bars_u + (warp * depth + slot) * 8;
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(bar, phase, err_u, p.status))) {
      ok = false;
      break;
    }
    // this lane's 32 packed bytes of rows g and g + 8, block tq (128-byte swizzle)
    const uint8_t *sb = smem + SL.ring + (warp * depth + slot) * kUnitBytes;
    const uint4 w0 = *reinterpret_cast<const uint4 *>(sb + g * 128 + (((2 * tq) ^ g) << 4));
    const uint4 w1 = *reinterpret_cast<const uint4 *>(sb + g * 128 + (((2 * tq + 1) ^ g) << 4));
    const uint4 v0 = *reinterpret_cast<const uint4 *>(sb + (g + 8) * 128 + (((2 * tq) ^ g) << 4));
    const uint4 v1 =
        *reinterpret_cast<const uint4 *>(sb + (g + 8) * 128 + (((2 * tq + 1) ^ g) << 4));
    ++done;
    const Nf4Table tg = make_table(ah_g, p.cb), th = make_table(ah_h, p.cb);
    const uint32_t wg[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
    const uint32_t wh[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    const uint4 *xlo = xr_lo + chunk * 32, *xhi = xr_hi + chunk * 32;
#pragma unroll
    for (int wi = 0; wi < 8; ++wi) {
      uint32_t og[4], oh[4];
      lookup8(tg, wg[wi], og);
      lookup8(th, wh[wi], oh);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const uint4 xv = (nt == 0 ? xlo : xhi)[xoff[wi]];
        mma_bf16(acc[nt], og[0], oh[0], og[1], oh[1], xv.x, xv.y);
        mma_bf16(acc[nt], og[2], oh[2], og[3], oh[3], xv.z, xv.w);
      }
    }
    // the slot's bytes are in registers and used: refill it with the unit
    // depth places ahead
    __syncwarp();
    if (lane == 0 && i + depth < u1 - u0) {
      fence_proxy_async_smem();
      issue(it_t, it_c, slot);
      step(it_t, it_c);
    }
    if (++slot == depth) {
      slot = 0;
      phase ^= 1u;
    }
    ah_g = nah_g;
    ah_h = nah_h;
    tile = ntile;
    chunk = nchunk;
  }
  if (ok && cur >= 0) flush(cur);
  if (!ok && lane == 0) {
    // error path: wait (bounded) for this warp's copies still in flight,
    // units done .. min(done + depth, count) - 1
    const int cnt = u1 - u0;
    for (int i = done; i < cnt && i < done + depth; ++i)
      mbar_drain(bars_u + (warp * depth + i % depth) * 8, (uint32_t)(i / depth) & 1u);
  }
  __syncthreads();

  // ---- 5. partial segments of each tile, added in warp order
  for (int i = threadIdx.x; i < Tc * 16 * MT; i += blockDim.x) {
    const int tile = i / (16 * MT), e = i - tile * 16 * MT;
    const int wa = wr[2 * tile], wb = wr[2 * tile + 1];
    if (wa == wb) continue;  // one warp covered the whole tile
    float v = 0.f;
    for (int w = wa; w <= wb; ++w) {
      const int sw = wr[2 * p.tiles_max + w];  // first tile of warp w
      v += part[(w * 2 + (sw == tile ? 0 : 1)) * 16 * MT + e];
    }
    tsum[tile * 16 * MT + e] = v;
  }
  cp_async_wait<0>();  // the B rows of the epilogue
  __syncthreads();
  cluster_sync();  // every CTA's tile sums are complete

  // ---- 6. t from the t kernel (the only input written by the kernel before)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  for (int i = threadIdx.x; i < p.M * p.RP; i += blockDim.x) tfin[i] = __ldcg(p.t + i);
  __syncthreads();
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // ---- 7. this CTA's share of the cluster's rows: y = sum over ranks + s t B^T
  {
    const uint32_t tsum_u = base + SL.tsum;
    const uint16_t *bsm = reinterpret_cast<const uint16_t *>(smem + SL.bs);
    // one (row, token) output per thread and pass, rows fastest
    for (int i = threadIdx.x; i < nr * p.M; i += blockDim.x) {
      const int m = i / nr, rl = r_lo + (i - m * nr);
      const int n = row0 + rl;
      const uint16_t *brow = bsm + (rl - r_lo) * p.r;
      const uint32_t off = tsum_u + ((rl >> 4) * 16 * MT + (rl & 15) * MT + m) * 4;
      float v = 0.f;
      for (int q = 0; q < S; ++q) v += ld_dsmem_f32(off, (uint32_t)q);
      float l = 0.f;
      const float *tc = tfin + m * p.RP;
      for (int c = 0; c < p.r; c += 8) {
        const uint4 bw = *reinterpret_cast<const uint4 *>(brow + c);
        l = fmaf(tc[c + 0], bf16_lo(bw.x), l);
        l = fmaf(tc[c + 1], bf16_hi(bw.x), l);
        l = fmaf(tc[c + 2], bf16_lo(bw.y), l);
        l = fmaf(tc[c + 3], bf16_hi(bw.y), l);
        l = fmaf(tc[c + 4], bf16_lo(bw.z), l);
        l = fmaf(tc[c + 5], bf16_hi(bw.z), l);
        l = fmaf(tc[c + 6], bf16_lo(bw.w), l);
        l = fmaf(tc[c + 7], bf16_hi(bw.w), l);
      }
      const float y = fmaf(p.s, l, v);
      const int64_t o = (int64_t)m * p.N + n;
      if (p.y_bf16)
        reinterpret_cast<__nv_bfloat16 *>(p.y)[o] = __float2bfloat16_rn(y);
      else
        reinterpret_cast<float *>(p.y)[o] = y;
    }
  }
  cluster_sync();  // keep this CTA's tile sums alive until the peers have read them
}

// ------------------------------------------------------------ launchers
// Largest dynamic shared memory of a GEMV CTA; set once on both instances so
// that the occupancy query and the launch see the same limit.
static constexpr int kGemvSmemMax = 232448;

static cudaError_t gemv_smem_attr() {
  static bool set = false;
  if (set) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(qlora_gemv_kernel<1>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kGemvSmemMax);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(qlora_gemv_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kGemvSmemMax);
  if (e != cudaSuccess) return e;
  set = true;
  return cudaSuccess;
}

// Clusters of S CTAs (smem bytes each) that the device runs at once: a
// cluster never spans two GPCs, so S * this can be below the SM count.
static int gemv_resident_clusters(int nt, int S, int smem, int want) {
  if (gemv_smem_attr() != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(want * S, 1, 1);
  cfg.blockDim = dim3(kGemvWarps * 32, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = S;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  const cudaError_t e =
      nt == 2 ? cudaOccupancyMaxActiveClusters(&n, qlora_gemv_kernel<2>, &cfg)
              : cudaOccupancyMaxActiveClusters(&n, qlora_gemv_kernel<1>, &cfg);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return n;
}

// Cluster size S (CTAs per cluster, each taking a slice of K) and the cluster
// count: S minimises the 2 KB units on the busiest CTA, ceil(tiles / clusters)
// x ceil(chunks / S), among the S whose shared memory fits, with the cluster
// count cut to what the device holds at once (one wave); ties go to the
// smaller S.
static int gemv_plan_uncached(int N, int K, int M, int r, int num_sms, GemvPlan *out);

// The plan depends on the shape and the device only; the occupancy queries
// behind it cost host time, so recent plans are kept (a small ring, under a
// lock: the library may be called from several host threads).
int gemv_plan(int N, int K, int M, int r, int num_sms, GemvPlan *out) {
  struct Entry {
    int N, K, M, r, num_sms, dev, rc;
    GemvPlan plan;
  };
  static std::mutex mu;
  static Entry cache[16];
  static int filled = 0, next = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < filled; ++i) {
      const Entry &e = cache[i];
      if (e.N == N && e.K == K && e.M == M && e.r == r && e.num_sms == num_sms && e.dev == dev) {
        if (out && e.rc == 0) *out = e.plan;
        return e.rc;
      }
    }
  }
  GemvPlan plan{};
  const int rc = gemv_plan_uncached(N, K, M, r, num_sms, &plan);
  {
    std::lock_guard<std::mutex> lock(mu);
    cache[next] = Entry{N, K, M, r, num_sms, dev, rc, plan};
    next = (next + 1) % 16;
    if (filled < 16) ++filled;
  }
  if (out && rc == 0) *out = plan;
  return rc;
}

static int gemv_plan_uncached(int N, int K, int M, int r, int num_sms, GemvPlan *out) {
  if (M < 1 || M > 16 || N < 1 || K < 64 || r < 1 || r > 64) return -1;
  if ((int64_t)N * (K / 64) >= ((int64_t)1 << 31)) return -1;  // 32-bit block indices
  const int RP = (r + 15) & ~15;
  const int MT = M > 8 ? 16 : 8;
  const int nt = M > 8 ? 2 : 1;
  const int T = (N + 15) / 16;
  const int C = (K + kChunk - 1) / kChunk;
  GemvPlan best{};
  int64_t best_load = -1;
  for (int S = 1; S <= 8; ++S) {
    const int sc = (C + S - 1) / S;
    if ((S - 1) * sc >= C) continue;  // every rank gets chunks
    for (int depth = kGemvDepthMax; depth >= 2; --depth) {
      int clusters = num_sms / S;
      if (clusters > T) clusters = T;
      if (clusters < 1) break;
      int tiles_max = 0, smem = 0;
      bool fits = false;
      for (int pass = 0; pass < 4 && clusters >= 1; ++pass) {
        tiles_max = (T + clusters - 1) / clusters;
        smem = gemv_smem(M, MT, sc, tiles_max, RP, depth, S).total;
        if (smem > kGemvSmemMax) break;
        const int res = gemv_resident_clusters(nt, S, smem, clusters);
        if (res >= clusters) {
          fits = true;
          break;
        }
        clusters = res;
      }
      if (!fits) continue;
      // a shallower ring only when the deeper one does not fit
      const int64_t load = (int64_t)tiles_max * sc;
      if (best_load < 0 || load < best_load) {
        best_load = load;
        best.S = S;
        best.slice_chunks = sc;
        best.clusters = clusters;
        best.tiles_total = T;
        best.tiles_max = tiles_max;
        best.smem = smem;
        best.depth = depth;
      }
      break;
    }
  }
  if (best_load < 0) return -1;
  if (out) *out = best;
  return 0;
}

cudaError_t launch_gemv(const CUtensorMap &tmW, GemvArgs a, const GemvPlan &plan,
                        const uint16_t *A, float *tpart, int *counter, float *t_save,
                        cudaStream_t s) {
  a.S = plan.S;
  a.slice_chunks = plan.slice_chunks;
  a.clusters = plan.clusters;
  a.tiles_total = plan.tiles_total;
  a.tiles_max = plan.tiles_max;
  a.depth = plan.depth;
  // t = x A^T into the workspace (a.t), partials in tpart
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((a.K + kChunk - 1) / kChunk, 1, 1);
    cfg.blockDim = dim3(kTWarps * 32, 1, 1);
    cfg.stream = s;
    cudaLaunchAttribute at[1] = {pdl_attr()};
    cfg.attrs = at;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, lora_t_decode_kernel, a.x, a.M, a.K, A, a.r, a.RP,
                                       tpart, const_cast<float *>(a.t), counter, t_save, a.mask,
                                       a.wpr, a.mask ? a.keep_scale : 1.0f);
    if (e != cudaSuccess) return e;
  }
  const int nt = a.M > 8 ? 2 : 1;
  cudaError_t e = gemv_smem_attr();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(plan.clusters * plan.S, 1, 1);
  cfg.blockDim = dim3(kGemvWarps * 32, 1, 1);
  cfg.dynamicSmemBytes = plan.smem;
  cfg.stream = s;
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = plan.S;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  attrs[1] = pdl_attr();
  cfg.attrs = attrs;
  cfg.numAttrs = 2;
  if (nt == 2)
    e = cudaLaunchKernelEx(&cfg, qlora_gemv_kernel<2>, tmW, a);
  else
    e = cudaLaunchKernelEx(&cfg, qlora_gemv_kernel<1>, tmW, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace qlora
