// merge.cu -- adapter merge for sm_103a:
//   W_out[n, k] = bf16_rn( w_hat[n, k] + s . sum_j B[n, j] A[j, k] ),  s = alpha / r
// ("QLoRA and 4bit Quantization | QLoRA 与 4-bit 量化", Step 5 conclusion:
// the merged adapter is what deployment loads; the forward formula of Step 3
// gives x W_hat^T + s (x A^T) B^T = x (W_hat + s B A)^T).
//
// HBM-bound (0.5 packed + 2 output bytes per weight).  Units of 16 rows x 256
// columns (4 blocks of 64); one wave of CTAs (as many as are resident), each
// taking an equal contiguous share of the units in chunk-major order.  The 8
// warps of a CTA take the row tiles of one 256-column chunk in turn, loading
// the next tile's packed bytes, block constants and B rows while they compute
// the current one; the chunk of A is staged once per chunk in shared memory
// (a CTA meets one or two chunks), while each warp's first loads are in
// flight.
//   - w_hat: lane (g, tq) dequantises rows g and g+8 of block tq with the
//     per-block byte-permute table (the dequantiser's routine: exact bf16),
//     its shifts on the multiply pipe (the integer pipe is the busier one).
//   - B A: bf16 mma.sync m16n8k16 (fp32 accumulation), A-operand = 16 rows
//     of B, B-operand = A.  The columns of n-tile j are mapped to positions
//     2j, 2j+1 of each lane group's block (column c -> block c / 2, position
//     2j + c % 2), so a lane's accumulator holds exactly the positions whose
//     w_hat pair its table lookup produced.
//   - A chunk in shared memory as [256 columns][RP ranks] bf16 with the
//     ranks of a row interleaved (0 1 8 9 2 3 10 11 ...) so that a lane's two
//     B-operand words are one 8-byte load.
//   - epilogue: fp32 w_hat + s . (B A), one rounding to bf16, into the warp's
//     8 KB staging tile in shared memory (the 128-byte swizzle of a tensor
//     map: 16-byte chunk q of 128-byte line L at L . 128 + (q ^ (L & 7)) . 16,
//     which keeps the eight lanes of each store phase on distinct banks), then
//     one TMA tensor store of the 16 x 256 tile (rows past N and blocks past
//     K / 64 are clipped by the copy).  Storing each lane's 16 bytes straight
//     to global memory instead touches 32 rows' lines per instruction and
//     took twice as long.
#include "common.cuh"
#include "kernels.h"

namespace qlora {

constexpr int kMergeWarps = 8;
constexpr int kMergeTileBytes = 16 * 256 * 2;  // one warp's staged output tile

// Dynamic shared memory of the kernel: the warps' output tiles (1024-byte
// aligned for the swizzle; 1024 bytes of slack), then the A chunk.
static int merge_smem_bytes(int ks) {
  return 1024 + kMergeWarps * kMergeTileBytes + 256 * ks * 16 * 2;
}

// A plain register function (no volatile), so that the compiler can
// interleave the MMAs with the loads and the table lookups.
__device__ __forceinline__ void mma_bf16_m(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                           uint32_t a3, uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Position of rank j inside an interleaved group of 16: 0 1 8 9 2 3 10 11 ...
__device__ __forceinline__ int rank_slot(int j) {
  const int q = j & 15;
  return (j & ~15) | (((q & 7) >> 1) << 2) | ((q >> 3) << 1) | (q & 1);
}

template <int KS>  // KS = RP / 16 rank steps
__global__ void __launch_bounds__(kMergeWarps * 32)
    merge_lora_kernel(const __grid_constant__ CUtensorMap tmO, const MergeArgs p) {
  extern __shared__ uint8_t msm_raw[];
  const uint32_t raw_u = smem_u32(msm_raw);
  const uint32_t tiles_u = (raw_u + 1023u) & ~1023u;
  uint16_t *as = reinterpret_cast<uint16_t *>(msm_raw + (tiles_u - raw_u) +
                                              kMergeWarps * kMergeTileBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t obuf = tiles_u + warp * kMergeTileBytes;
  const int g = lane >> 2, tq = lane & 3;
  constexpr int RP = KS * 16;
  const int kbr = p.K >> 6;
  const int ntiles = (p.N + 15) / 16;
  // this CTA's units: [u0, u1) of the chunk-major (chunk, row tile) order
  const int64_t units = (int64_t)((p.K + 255) / 256) * ntiles;
  const int64_t u0 = units * blockIdx.x / gridDim.x, u1 = units * (blockIdx.x + 1) / gridDim.x;
  // packed bytes, block constant and B fragments of one tile's rows n0, n1
  struct TileIn {
    uint4 l0, h0, l1, h1;
    float ah0, ah1;
    uint32_t af[KS][4];
  };
  auto fetch = [&](int blk, int tile, TileIn &d) {
    const bool kin = blk < kbr;
    const int n0 = tile * 16 + g, n1 = n0 + 8;
    auto one = [&](int n, uint4 &lo, uint4 &hi, float &ahat) {
      const bool ok = kin && n < p.N;
      const int64_t b64 = ok ? (int64_t)n * kbr + blk : 0;  // clamped into the arrays
      const uint8_t *src = p.packed + b64 * 32;
      lo = ldg_nc_v4(src);
      hi = ldg_nc_v4(src + 16);
      const int64_t b = b64 >> p.bshift;
      const float cv = ldg_nc_f32(p.cvec + (b >> p.cshift));
      const float a = p.use_code ? __fmul_rn((float)ldg_nc_s8(p.codes + b), cv) : cv;
      ahat = ok ? a : 0.f;
    };
    one(n0, d.l0, d.h0, d.ah0);
    one(n1, d.l1, d.h1, d.ah1);
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const int j0 = ks * 16 + 2 * tq;
      auto bw = [&](int n, int j) -> uint32_t {
        if (n >= p.N || j >= p.r) return 0u;
        return __ldg(reinterpret_cast<const uint32_t *>(p.B + (int64_t)n * p.r + j));
      };
      d.af[ks][0] = bw(n0, j0);
      d.af[ks][1] = bw(n1, j0);
      d.af[ks][2] = bw(n0, j0 + 8);
      d.af[ks][3] = bw(n1, j0 + 8);
    }
  };
  // this lane's column of every n-tile: block g >> 1, position 2j + (g & 1)
  const int bcol = (g >> 1) * 64 + (g & 1);
  // 128-byte lines of rows g and g + 8 in block tq (same swizzle: 32 lines apart)
  const uint32_t line0 = g * 4 + tq;
  const uint32_t row0_u = obuf + line0 * 128, row1_u = row0_u + 32 * 128;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  for (int chunk = (int)(u0 / ntiles); (int64_t)chunk * ntiles < u1; ++chunk) {
    const int64_t cbase = (int64_t)chunk * ntiles;
    const int lo = (int)((u0 > cbase ? u0 : cbase) - cbase);
    const int hi = (int)((u1 < cbase + ntiles ? u1 : cbase + ntiles) - cbase);
    const int kc0 = chunk * 256;
    const int blk = chunk * 4 + tq;  // 64-chunk of the row
    int tile = lo + warp;
    TileIn cur;
    if (tile < hi) fetch(blk, tile, cur);  // in flight while A is staged
    __syncthreads();  // the previous chunk's A is no longer read
    // A chunk -> shared memory, transposed and rank-interleaved (0 past r or
    // K): 16-byte loads of 8 columns of one rank, scattered to the 8 columns
    for (int i = threadIdx.x; i < 32 * RP; i += blockDim.x) {
      const int j = i / 32, c8 = (i - j * 32) * 8;
      const int k = kc0 + c8;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (j < p.r && k < p.K) v = ldg_nc_v4(p.A + (int64_t)j * p.K + k);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      const int sl = rank_slot(j);
#pragma unroll
      for (int e = 0; e < 8; ++e)
        as[(c8 + e) * RP + sl] = (uint16_t)(w[e >> 1] >> ((e & 1) * 16));
    }
    __syncthreads();
    for (; tile < hi; tile += kMergeWarps) {
      // the next tile's loads are in flight while this one is computed
      TileIn nxt;
      const bool more = tile + kMergeWarps < hi;
      if (more) fetch(blk, tile + kMergeWarps, nxt);
      const Nf4Table t0 = make_table(cur.ah0, p.cb), t1 = make_table(cur.ah1, p.cb);
      // the previous tile's store has read the staging tile
      if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
      __syncwarp();
      const uint32_t w0[8] = {cur.l0.x, cur.l0.y, cur.l0.z, cur.l0.w,
                              cur.h0.x, cur.h0.y, cur.h0.z, cur.h0.w};
      const uint32_t w1[8] = {cur.l1.x, cur.l1.y, cur.l1.z, cur.l1.w,
                              cur.h1.x, cur.h1.y, cur.h1.z, cur.h1.w};
#pragma unroll
      for (int wi = 0; wi < 8; ++wi) {
        uint32_t o0[4], o1[4];
        lookup8_mulhi(t0, w0[wi], o0, p.k31, p.k16);
        lookup8_mulhi(t1, w1[wi], o1, p.k31, p.k16);
        uint32_t r0[4], r1[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int j = wi * 4 + q;  // n-tile: positions 2j, 2j + 1
          float d[4] = {0.f, 0.f, 0.f, 0.f};
          const uint2 *arow = reinterpret_cast<const uint2 *>(as + (bcol + 2 * j) * RP + tq * 4);
#pragma unroll
          for (int ks = 0; ks < KS; ++ks) {
            const uint2 bv = arow[ks * 4];  // 16 ranks = 32 bytes = 4 uint2 per step
            mma_bf16_m(d, cur.af[ks][0], cur.af[ks][1], cur.af[ks][2], cur.af[ks][3], bv.x, bv.y);
          }
          r0[q] = pack_bf16x2(fmaf(p.s, d[0], bf16_lo(o0[q])), fmaf(p.s, d[1], bf16_hi(o0[q])));
          r1[q] = pack_bf16x2(fmaf(p.s, d[2], bf16_lo(o1[q])), fmaf(p.s, d[3], bf16_hi(o1[q])));
        }
        const uint32_t q16 = (wi ^ (line0 & 7)) << 4;
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(row0_u + q16), "r"(r0[0]),
                     "r"(r0[1]), "r"(r0[2]), "r"(r0[3]) : "memory");
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(row1_u + q16), "r"(r1[0]),
                     "r"(r1[1]), "r"(r1[2]), "r"(r1[3]) : "memory");
      }
      fence_proxy_async_smem();  // the tile's generic-proxy writes, before the async store
      __syncwarp();
      if (lane == 0) {
        asm volatile(
            "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];"
            ::"l"(reinterpret_cast<uint64_t>(&tmO)), "r"(0), "r"(chunk * 4), "r"(tile * 16),
            "r"(obuf)
            : "memory");
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
      }
      if (more) cur = nxt;
    }
  }
  // every store of the warp complete before the CTA ends
  if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

cudaError_t launch_merge(const CUtensorMap &tmO, const MergeArgs &a, int num_sms,
                         cudaStream_t s) {
  if (a.N == 0 || a.K == 0) return cudaSuccess;
  static bool attr_set[5] = {false, false, false, false, false};
  const int64_t units = (int64_t)((a.N + 15) / 16) * ((a.K + 255) / 256);
  static int occ[5] = {0, 0, 0, 0, 0};  // resident CTAs per SM of each instance
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kMergeWarps * 32, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute at[1] = {pdl_attr()};
  cfg.attrs = at;
  cfg.numAttrs = 1;
  const int ks = (a.r + 15) / 16;
  if (ks < 1 || ks > 4) return cudaErrorInvalidValue;
  cfg.dynamicSmemBytes = merge_smem_bytes(ks);
  auto go = [&](auto kern) -> cudaError_t {
    if (!attr_set[ks]) {
      const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)cfg.dynamicSmemBytes);
      if (e != cudaSuccess) return e;
      attr_set[ks] = true;
      int n = 0;
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kMergeWarps * 32,
                                                    cfg.dynamicSmemBytes);
      occ[ks] = n > 0 ? n : 1;
    }
    // one wave, and no more CTAs than one per 8 units
    const int64_t want = (units + kMergeWarps - 1) / kMergeWarps;
    const int64_t cap = (int64_t)num_sms * occ[ks];
    cfg.gridDim = dim3((unsigned)(want < cap ? want : cap), 1, 1);
    return cudaLaunchKernelEx(&cfg, kern, tmO, a);
  };
  switch (ks) {
    case 1: return go(merge_lora_kernel<1>);
    case 2: return go(merge_lora_kernel<2>);
    case 3: return go(merge_lora_kernel<3>);
    case 4: return go(merge_lora_kernel<4>);
  }
  return cudaErrorInvalidValue;
}

}  // namespace qlora
