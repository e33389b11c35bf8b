// quantize.cu -- blockwise NF4 quantisation with double quantisation, and
// dequantisation to bf16, for sm_103a.
//
// Method ("第 09 期 | QLoRA 4-bit 量化微调" section 9.2.1-9.2.2; "QLoRA and 4bit
// Quantization | QLoRA 与 4-bit 量化" Step 2; "QLoRA 的三个核心技术", double
// quantization): each 64-weight block is normalised by its absolute maximum,
// every normalised weight becomes the 4-bit index of its nearest NF4
// codepoint, two indices share a byte, and the block maxima are quantised
// again to int8 with one fp32 scale per group of block constants.
//
// Both kernels stream the weight through HBM once; the quantiser is limited
// by instruction issue, the dequantiser by the integer pipe (the byte
// permutes).  Layout of the work:
//   quantise: persistent CTAs of 512 (+ 32) or 1024 threads, each taking groups of 256
//     consecutive blocks (one double quantisation group of 256, or several
//     smaller groups), the input of each group brought into shared memory
//     by one bulk copy a few groups ahead.  Eight lanes share a block
//     (sixteen for 128-weight blocks): each lane reads 16 bytes of bf16 (or
//     32 of fp32), the block maximum is a shuffle reduction, and the lane
//     writes its 8 indices as one 32-bit word, so each warp instruction
//     moves 512 contiguous bytes in and 128 contiguous bytes out.
//   dequantise: four lanes per block, 16 elements per lane; the per-block
//     scaled table T[i] = bf16(c_i * a_hat) is built once per lane and
//     indexed with byte permutes (the same routine the fused GEMM producer
//     uses), 32-byte stores.
#include <cmath>

#include "common.cuh"
#include "kernels.h"

namespace qlora {

// Decision tables of the nearest-codepoint rule (built on the host from the
// 15 thresholds; see launch_quantize):
//   th[k]     the thresholds: index = #{k : x >= th[k]} (th[15] = 2)
//   for the 1/16-wide bucket i of [-1, 1] (x in [-1 + i/16, -1 + (i + 1)/16),
//   i = -1 .. 32), at slot i + 1:
//   nth[]     minus the one threshold inside the bucket (-2 when there is
//             none)
//   base1[]   one more than the number of thresholds below the bucket
// (two 34-word arrays: a warp's lookups then meet no bank conflict unless two
// lanes hold elements near -1 and near +1 at once)
struct QuantTables {
  float th[16];
  float nth[34];
  int base1[34];
  int exact_only;  // 1: some bucket holds two thresholds; divide every element
};

// Number of thresholds <= x, by bisection over the sorted thresholds.
__device__ __forceinline__ int nf4_index(float x, const float *th) {
  int i = (x >= th[7]) ? 8 : 0;
  i += (x >= th[i + 3]) ? 4 : 0;
  i += (x >= th[i + 1]) ? 2 : 0;
  i += (x >= th[i]) ? 1 : 0;
  return i;
}

// Byte offset of element e (0..7) of a lane's 8 consecutive elements in its
// packed 32-bit word: byte e/2, element 2j in the high nibble.
__device__ __forceinline__ constexpr int nib_shift(int e) { return 8 * (e >> 1) + ((e & 1) ? 0 : 4); }

// Band (absolute, in normalised units) around each threshold inside which
// the reciprocal-based decision may differ from the one on the IEEE quotient.
// With y the hardware reciprocal (rcp.approx: at most 1 ulp from 1/a, so
// y = (1/a)(1 + d1) with |d1| <= 2^-23 for a normal a and y), the fast path
// compares the exact product z = w y (inside an FMA) with th:
//   z = (w/a)(1 + d1),  RN(w/a) = (w/a)(1 + d3),  |d3| <= 2^-24,
// so |z - RN(w/a)| < 2^-22.4 |w/a| <= 2^-22.4.  If [z >= th] and
// [RN(w/a) >= th] differ, then |z - th| < 2^-22.4 (th is a float, so
// RN(w/a) < th means RN(w/a) <= pred(th) and z < th + 2^-22.4; RN(w/a) >= th
// means z > th - 2^-22.4), so every element whose |RN(z - th)| is at least
// 2^-20 is decided the same way by both.
constexpr float kQuantBand = 9.5367431640625e-07f;  // 2^-20

// kR = block / 64.  A CTA of T threads takes groups of 256 consecutive
// blocks (one double-quantisation group of 256, or several smaller groups):
// group g, g + gridDim.x, ... (persistent grid).  Pass p, warp w, lane group
// `sub` (8 lanes) covers 64-element chunk p * T / 8 + 4 w + sub of the group,
// lane li its elements 8 li .. 8 li + 7; the 8 kR lanes of a block reduce its
// maximum with shuffles.
//
// kBulk: the group's input (contiguous, 32 kR KB of bf16 or 64 kR KB of fp32)
// comes into one of kQStages shared-memory stages with a single bulk copy
// (cp.async.bulk, completion on the stage's mbarrier); one thread refills a
// stage as soon as every thread has read it (after a CTA-wide barrier, or,
// with the extra warp of the bf16 / 64 case, when the stage's "empty"
// mbarrier has the 16 pass warps' arrivals), so the next stages' copies are
// in flight while a group is computed.  Without kBulk (fp32 weights in
// 128-weight blocks: three 128 KB stages would not fit) every thread loads
// its pieces straight into registers.
constexpr int kQStages = 3;
template <bool kBf16In, int kR>
__host__ __device__ constexpr bool quant_bulk() { return kBf16In || kR == 1; }
// 32 pass warps per SM either way: bf16 weights in 64-weight blocks run two CTAs
// of 512 threads per SM (two 96 KB stage rings; half the warps at each
// barrier; each CTA with one more warp for the double quantisation), the
// other staged cases one CTA of 1024 threads (a 192 KB ring),
// and fp32 weights in 128-weight blocks, which hold all their pieces in
// registers, one CTA of 512.
template <bool kBf16In, int kR>
__host__ __device__ constexpr int quant_threads() {
  return (kBf16In && kR == 1) ? 512 : (quant_bulk<kBf16In, kR>() ? 1024 : 512);
}
// bf16 weights in 64-weight blocks: one more warp per CTA runs the double
// quantisation of each group while the 16 others start the next group.
template <bool kBf16In, int kR>
__host__ __device__ constexpr bool quant_dq_warp() { return kBf16In && kR == 1; }
template <bool kBf16In, int kR>
__host__ __device__ constexpr int quant_launch_threads() {
  return quant_threads<kBf16In, kR>() + (quant_dq_warp<kBf16In, kR>() ? 32 : 0);
}
template <bool kBf16In, int kR>
__host__ __device__ constexpr int quant_stage_bytes() { return 256 * kR * 64 * (kBf16In ? 2 : 4); }
template <bool kBf16In, int kR>
__host__ __device__ constexpr int quant_smem_bytes() {
  return quant_bulk<kBf16In, kR>() ? kQStages * quant_stage_bytes<kBf16In, kR>() + 128 : 0;
}

// (a minimum of 0 resident CTAs leaves the register budget of the other
// instances to the compiler, as without the bound)
template <bool kBf16In, int kR>
__global__ void __launch_bounds__(quant_launch_threads<kBf16In, kR>(),
                                  quant_dq_warp<kBf16In, kR>() ? 2 : 0)
    quantize_nf4_kernel(const void *__restrict__ W,
                                                             int64_t nblocks, int group,
                                                             uint8_t *__restrict__ packed,
                                                             int8_t *__restrict__ codes,
                                                             float *__restrict__ absf,
                                                             float *__restrict__ scale2,
                                                             int *__restrict__ nonfinite_flag,
                                                             const QuantTables tab) {
  extern __shared__ __align__(128) uint8_t qsm[];  // [stage][group input]; mbarriers at the end
  __shared__ float th_s[16];
  __shared__ uint32_t bt_s[68];  // nth[34] then base1[34]
  __shared__ float amax_s[2][256];  // block maxima of the last two groups
  __shared__ float wmax_s[8];
  __shared__ uint32_t qerr_s;
  constexpr bool kBulk = quant_bulk<kBf16In, kR>();
  constexpr int kStage = quant_stage_bytes<kBf16In, kR>();
  constexpr int kT = quant_threads<kBf16In, kR>();  // threads of the element passes
  constexpr bool kDqWarp = quant_dq_warp<kBf16In, kR>();
  constexpr int kCpp = kT / 8;                 // chunks per pass
  constexpr int kPasses = 256 * kR / kCpp;
  constexpr int kEsz = kBf16In ? 2 : 4;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int sub = lane >> 3, li = lane & 7;
  const int64_t nchunks = nblocks * kR;  // 64-element chunks
  const int64_t ngroups = (nblocks + 255) / 256;
  const int64_t G = gridDim.x;
  const uint32_t sm_u = smem_u32(qsm);
  const uint32_t bars_u = sm_u + kQStages * kStage;  // kQStages mbarriers (kBulk)
  if (tid < 16) th_s[tid] = tab.th[tid];
  if (tid < 34) {
    bt_s[tid] = __float_as_uint(tab.nth[tid]);
    bt_s[34 + tid] = (uint32_t)tab.base1[tid];
  }
  // mbarriers: full[kQStages] (the stage's copy landed); with the extra
  // warp also empty[kQStages] (every pass warp has read the stage),
  // amax_full[2] (every pass warp has written the group's block maxima) and
  // amax_free[2] (the extra warp has read them), which take the place of a
  // CTA-wide barrier per group
  if (kBulk && tid < kQStages) mbar_init(bars_u + tid * 8, 1);
  if (kDqWarp && tid < kQStages) mbar_init(bars_u + (kQStages + tid) * 8, kT / 32);
  if (kDqWarp && tid < 2) {
    mbar_init(bars_u + (2 * kQStages + tid) * 8, kT / 32);
    mbar_init(bars_u + (2 * kQStages + 2 + tid) * 8, 1);
  }
  if (tid == 0) qerr_s = 0u;
  if (kBulk) fence_barrier_init();
  __syncthreads();  // tables and barriers ready
  pdl_wait_release();  // every global access below follows the previous kernel

  // one bulk copy of group grp's input into stage st (thread 0)
  auto issue = [&](int64_t grp, int st) {
    const int64_t e0 = grp * 256 * kR * 64;
    const int64_t el = min((int64_t)256 * kR * 64, nchunks * 64 - e0);
    const uint32_t bytes = (uint32_t)(el * kEsz);  // a multiple of 128
    const uint32_t bar = bars_u + st * 8;
    mbar_arrive_expect_tx(bar, bytes);
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(sm_u + st * kStage),
        "l"(reinterpret_cast<const uint8_t *>(W) + e0 * kEsz), "r"(bytes), "r"(bar)
        : "memory");
  };
  if (kBulk && tid == 0)
    for (int st = 0; st < kQStages; ++st)
      if (blockIdx.x + st * G < ngroups) issue(blockIdx.x + st * G, st);
  // bounded wait (~2 s); past the limit the error is recorded and the work
  // goes on with whatever the buffers hold
  auto bwait = [&](uint32_t bar, uint32_t ph) {
    if (!mbar_try_wait(bar, ph)) {
      const long long t0 = clock64();
      while (!mbar_try_wait(bar, ph))
        if (clock64() - t0 > (1ll << 32)) {
          qerr_s = 1u;
          break;
        }
    }
  };
  const uint32_t empty_u = bars_u + kQStages * 8;       // empty[st]
  const uint32_t afull_u = bars_u + 2 * kQStages * 8;   // amax_full[b]
  const uint32_t afree_u = afull_u + 2 * 8;             // amax_free[b]

  int nonfinite = 0;
  int it = 0;
  for (int64_t grp = blockIdx.x; grp < ngroups; grp += G, ++it) {
    const int64_t blk0 = grp * 256;   // first block of the group
    const int64_t ch0 = blk0 * kR;    // its first 64-element chunk
    const int st = it % kQStages;
    if (!kDqWarp || warp < kT / 32) {  // the element passes
    constexpr int kWords = kBf16In ? 4 : 8;  // 32-bit words per pass
    uint32_t raw[kPasses][kWords];
    bool inb[kPasses];
    if constexpr (kBulk) {
      // bounded wait on the stage (~2 s); past the limit the group is
      // computed from whatever the stage holds and the error is reported
      bwait(bars_u + st * 8, (uint32_t)(it / kQStages) & 1u);
      const uint8_t *stg = qsm + st * kStage;
#pragma unroll
      for (int p = 0; p < kPasses; ++p) {
        const int c = p * kCpp + warp * 4 + sub;
        inb[p] = ch0 + c < nchunks;
        const uint4 *src = reinterpret_cast<const uint4 *>(stg + (c * 64 + li * 8) * kEsz);
        const uint4 u0 = src[0];
        raw[p][0] = u0.x, raw[p][1] = u0.y, raw[p][2] = u0.z, raw[p][3] = u0.w;
        if constexpr (!kBf16In) {
          const uint4 u1 = src[1];
          raw[p][4] = u1.x, raw[p][5] = u1.y, raw[p][6] = u1.z, raw[p][7] = u1.w;
        }
      }
      if constexpr (kDqWarp) {  // this warp is done with the stage
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_u + st * 8);
      }
    } else {
#pragma unroll
      for (int p = 0; p < kPasses; ++p) {
        const int c = p * kCpp + warp * 4 + sub;
        inb[p] = ch0 + c < nchunks;
        const uint8_t *src = reinterpret_cast<const uint8_t *>(W) +
                             ((inb[p] ? ch0 + c : 0) * 64 + li * 8) * kEsz;
        const uint4 u0 = inb[p] ? ldg_nc_v4(src) : make_uint4(0, 0, 0, 0);
        raw[p][0] = u0.x, raw[p][1] = u0.y, raw[p][2] = u0.z, raw[p][3] = u0.w;
        if constexpr (!kBf16In) {
          const uint4 u1 = inb[p] ? ldg_nc_v4(src + 16) : make_uint4(0, 0, 0, 0);
          raw[p][4] = u1.x, raw[p][5] = u1.y, raw[p][6] = u1.z, raw[p][7] = u1.w;
        }
      }
    }
    // chunks past the end of the weight (the stage holds stale bytes there)
    // count as zeros; only the last group has any
    if (grp == ngroups - 1) {
#pragma unroll
      for (int p = 0; p < kPasses; ++p)
        if (!inb[p])
#pragma unroll
          for (int q = 0; q < kWords; ++q) raw[p][q] = 0u;
    }

    auto elem = [&](int p, int e) -> float {
      if (kBf16In) return (e & 1) ? bf16_hi(raw[p][e >> 1]) : bf16_lo(raw[p][e >> 1]);
      return __uint_as_float(raw[p][e]);
    };
    // the extra warp has read the maxima of two groups ago from this buffer
    if (kDqWarp && it >= 2) bwait(afree_u + (it & 1) * 8, (uint32_t)((it >> 1) - 1) & 1u);

#pragma unroll
    for (int p = 0; p < kPasses; ++p) {
      const int c = p * kCpp + warp * 4 + sub;
      // Block absmax as the largest magnitude bit pattern (the order of
      // non-negative floats); a pattern >= 0x7f800000 means an infinite or NaN
      // element, and the maximum is then taken over the finite ones only.
      uint32_t mb;
      if (kBf16In) {
        // two magnitudes per instruction: max of |a|, |b| (the sign of the
        // result is not used), a NaN kept so that the test below sees it
        uint32_t m2 = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          asm("max.NaN.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m2) : "r"(raw[p][q]));
        m2 &= 0x7fff7fffu;
        mb = max(m2 << 16, m2 & 0xffff0000u);
      } else {
        mb = 0;
#pragma unroll
        for (int q = 0; q < 8; ++q) mb = max(mb, raw[p][q] & 0x7fffffffu);
      }
      mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
      mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
      mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, 4));
      if (kR == 2) mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, 8));
      const bool nf = mb >= 0x7f800000u;
      if (__any_sync(0xffffffffu, nf)) {  // rare: some block of the warp is not finite
        uint32_t mf = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint32_t bits = __float_as_uint(elem(p, e)) & 0x7fffffffu;
          if (bits < 0x7f800000u) mf = max(mf, bits);
        }
        mf = max(mf, __shfl_xor_sync(0xffffffffu, mf, 1));
        mf = max(mf, __shfl_xor_sync(0xffffffffu, mf, 2));
        mf = max(mf, __shfl_xor_sync(0xffffffffu, mf, 4));
        if (kR == 2) mf = max(mf, __shfl_xor_sync(0xffffffffu, mf, 8));
        if (nf) {
          mb = mf;
          ++nonfinite;
          // the block's non-finite elements become zeros (their indices are
          // unspecified), so that every element below is a finite |w| <= amax
#pragma unroll
          for (int q = 0; q < kWords; ++q) {
            uint32_t v = raw[p][q];
            if (kBf16In) {
              if ((v & 0x7f800000u) == 0x7f800000u) v &= 0x0000ffffu;
              if ((v & 0x00007f80u) == 0x00007f80u) v &= 0xffff0000u;
            } else if ((v & 0x7f800000u) == 0x7f800000u) {
              v = 0u;
            }
            raw[p][q] = v;
          }
        }
      }
      const float amax = __uint_as_float(mb);
      if (li == 0 && (sub % kR) == 0) amax_s[it & 1][c / kR] = amax;  // 0 past the end
      // Fast path: y the hardware reciprocal of a (within 1 ulp of 1/a);
      // the bucket of z = w y and its threshold test are one FMA each, and
      // an element whose test lies within the band is decided again with
      // the IEEE quotient.  Block constants outside [2^-120, 2^120] take the
      // IEEE path for every element (y = 0 keeps their buckets in range).
      const bool fast = !tab.exact_only && amax >= 0x1p-120f && amax <= 0x1p120f;
      float y;
      asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(amax));
      y = fast ? y : 0.0f;
      const float y16 = y * 16.0f;
      // u = RD(16 w y + 16 + 1.5 . 2^23) = 1.5 . 2^23 + i, i = floor(16 z + 16)
      // in [-1, 32] (|w| <= a), exactly (one rounding, toward -inf, to the
      // integers); the bit pattern of u is 0x4b400000 + i, so nth[i + 1]
      // lies at bits(u) . 4 + (bt_s + 4 - 0x4b400000 . 4), modulo 2^32, and
      // base1[i + 1] 136 bytes further.  Both FMAs take the lane's elements
      // in pairs (packed f32x2: the two halves are rounded independently).
      const uint32_t tb = smem_u32(bt_s) + 4u - 0x2d000000u;
      // word = sum of base1_e << nib_shift(e) minus the sign bits of the d_e
      // at the same places (each nibble base1 - [d < 0] is in 0..15, so the
      // difference is the packed word; borrows cancel across the sum)
      uint32_t word = 0;
      float dmin = 1.0f;  // smallest |z - th| of the lane's elements
      uint32_t db[8];     // bit patterns of the d_e
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        const float w0 = elem(p, e), w1 = elem(p, e + 1);
        float u0, u1;
        asm("{.reg .b64 rw, ry, rc, rd;\n\tmov.b64 rw, {%2, %3};\n\tmov.b64 ry, {%4, %4};\n\t"
            "mov.b64 rc, {%5, %5};\n\tfma.rm.f32x2 rd, rw, ry, rc;\n\tmov.b64 {%0, %1}, rd;}"
            : "=f"(u0), "=f"(u1) : "f"(w0), "f"(w1), "f"(y16), "f"(12582928.0f));
        uint32_t t0, b0, t1, b1;
        asm("ld.shared.u32 %0, [%2];\n\tld.shared.u32 %1, [%2+136];"
            : "=r"(t0), "=r"(b0) : "r"(__float_as_uint(u0) * 4u + tb));
        asm("ld.shared.u32 %0, [%2];\n\tld.shared.u32 %1, [%2+136];"
            : "=r"(t1), "=r"(b1) : "r"(__float_as_uint(u1) * 4u + tb));
        // d = RN(z - th): non-negative exactly when z >= th (a zero is +0),
        // so the index is base1 - [d < 0]
        float d0, d1;
        asm("{.reg .b64 rw, ry, rt, rd;\n\tmov.b64 rw, {%2, %3};\n\tmov.b64 ry, {%4, %4};\n\t"
            "mov.b64 rt, {%5, %6};\n\tfma.rn.f32x2 rd, rw, ry, rt;\n\tmov.b64 {%0, %1}, rd;}"
            : "=f"(d0), "=f"(d1) : "f"(w0), "f"(w1), "f"(y), "r"(t0), "r"(t1));
        dmin = fminf(dmin, fminf(fabsf(d0), fabsf(d1)));
        word += b0 << nib_shift(e);
        word += b1 << nib_shift(e + 1);
        db[e] = __float_as_uint(d0);
        db[e + 1] = __float_as_uint(d1);
      }
      {
        // sign-replicating byte permutes: byte j of se is 0xff when d_{2j} < 0,
        // of so when d_{2j+1} < 0
        const uint32_t se = prmt(prmt(db[0], db[2], 0x00FBu), prmt(db[4], db[6], 0xFB00u), 0x7610u);
        const uint32_t so = prmt(prmt(db[1], db[3], 0x00FBu), prmt(db[5], db[7], 0xFB00u), 0x7610u);
        word -= (se & 0x10101010u) | (so & 0x01010101u);
      }
      // The vote is taken by every lane of the warp (lanes of all-zero
      // blocks and of blocks past the end included), outside any branch.
      const bool redo = amax != 0.0f && (dmin < kQuantBand || !fast);
      if (__any_sync(0xffffffffu, redo) && redo) {
        word = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e)
          word |= (uint32_t)nf4_index(__fdiv_rn(elem(p, e), amax), th_s) << nib_shift(e);
      }
      if (amax == 0.0f) word = 0x77777777u;  // every index is the exact-zero codepoint
      if (inb[p]) *reinterpret_cast<uint32_t *>(packed + (ch0 + c) * 32 + li * 4) = word;
    }
    if constexpr (kDqWarp) {  // this warp's block maxima of the group are written
      __syncwarp();
      if (lane == 0) mbar_arrive(afull_u + (it & 1) * 8);
    }
    }
    if constexpr (!kDqWarp) {
      __syncthreads();  // amax_s[it & 1] complete; every thread is done with the stage
      if (kBulk && tid == 0 && grp + kQStages * G < ngroups) {
        fence_proxy_async_smem();
        issue(grp + kQStages * G, st);
      }
    }

    // Second level: one scale per `group` consecutive block constants, by
    // threads 0..255 (warps 0..7), while the other warps go on to the next
    // group: the block maxima are double-buffered, and the 8 warps meet at a
    // barrier of their own (the next CTA-wide barrier, after the next group's
    // elements, orders this step before the buffers are reused).
    if (kDqWarp) {
      // the extra warp: it refills the stage once every pass warp has read
      // it, then, once they have all written the group's block maxima, runs
      // the double quantisation (lane L: blocks 8L .. 8L + 7, whose group
      // spans group / 8 consecutive lanes) and frees the maxima buffer
      if (warp == kT / 32) {
        if (grp + kQStages * G < ngroups) {
          if (lane == 0) {
            bwait(empty_u + st * 8, (uint32_t)(it / kQStages) & 1u);
            fence_proxy_async_smem();
            issue(grp + kQStages * G, st);
          }
          __syncwarp();
        }
        bwait(afull_u + (it & 1) * 8, (uint32_t)(it >> 1) & 1u);
        const float *am = amax_s[it & 1];
        float a[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) a[j] = am[8 * lane + j];
        const int64_t gb0 = blk0 + 8 * lane;
        if (group == 0) {
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (gb0 + j < nblocks) absf[gb0 + j] = a[j];
        } else {
          float m = a[0];
#pragma unroll
          for (int j = 1; j < 8; ++j) m = fmaxf(m, a[j]);
          for (int o = 1; o < (group >> 3); o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
          const float s2 = __fdiv_rn(m, 127.0f);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            float c = 0.0f;
            if (s2 != 0.0f) c = rintf(__fdiv_rn(a[j], s2));
            c = fminf(fmaxf(c, -127.0f), 127.0f);
            if (gb0 + j < nblocks) codes[gb0 + j] = (int8_t)(int)c;
          }
          if (((8 * lane) & (group - 1)) == 0 && gb0 < nblocks) scale2[gb0 / group] = s2;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(afree_u + (it & 1) * 8);
      }
    } else if (tid < 256) {
      const float a = amax_s[it & 1][tid];
      const int64_t gb = blk0 + tid;
      if (group == 0) {
        if (gb < nblocks) absf[gb] = a;
      } else {
        float m = a;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) wmax_s[warp] = m;
        asm volatile("bar.sync 1, 256;" ::: "memory");
        const int wpg = group >> 5;  // warps per group (group >= 32)
        const int w0 = (warp / wpg) * wpg;
        float gmax = 0.0f;
        for (int w = w0; w < w0 + wpg; ++w) gmax = fmaxf(gmax, wmax_s[w]);
        const float s2 = __fdiv_rn(gmax, 127.0f);
        float c = 0.0f;
        if (s2 != 0.0f) c = rintf(__fdiv_rn(a, s2));
        c = fminf(fmaxf(c, -127.0f), 127.0f);
        if (gb < nblocks) {
          codes[gb] = (int8_t)(int)c;
          if ((tid % group) == 0) scale2[gb / group] = s2;
        }
      }
    }
  }
  __syncthreads();  // every warp done (a timeout of any of them is in qerr_s)
  if (nonfinite_flag) {
    nonfinite = __any_sync(0xffffffffu, nonfinite != 0);
    if (nonfinite && lane == 0) atomicExch(nonfinite_flag, 1);
    if (tid == 0 && qerr_s) atomicExch(nonfinite_flag, kStatusTimeout);
  }
}

// ------------------------------------------------------------- dequantise
__global__ void __launch_bounds__(256) dequant_nf4_kernel(const uint8_t *__restrict__ packed,
                                                          const int8_t *__restrict__ codes,
                                                          const float *__restrict__ absf,
                                                          const float *__restrict__ scale2,
                                                          int group, int64_t npieces,
                                                          int piece_shift,
                                                          uint16_t *__restrict__ out,
                                                          const Codebook cb) {
  pdl_wait_release();
  // piece q (16 elements) lies in block q >> piece_shift (block / 16 pieces)
  for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < npieces;
       q += (int64_t)gridDim.x * blockDim.x) {
    const int64_t b = q >> piece_shift;
    const uint2 pk = ldg_nc_v2(packed + q * 8);
    float ahat;
    if (group > 0)
      ahat = __fmul_rn((float)codes[b], scale2[b / group]);
    else
      ahat = absf[b];
    const Nf4Table t = make_table(ahat, cb);
    uint32_t o[8];
    lookup8(t, pk.x, o);
    lookup8(t, pk.y, o + 4);
    uint4 *dst = reinterpret_cast<uint4 *>(out + q * 16);
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

// ----------------------------------------------------------- host launchers
// Bucket tables for the fast decision path, from the 15 sorted thresholds.
// The bucket of an element is found exactly, so the tables are valid when no
// 1/16-wide bucket holds two thresholds (true of both codebooks, whose
// thresholds lie more than 1/16 apart); otherwise every element is divided.
static void build_quant_tables(const float th[15], QuantTables &t) {
  for (int i = 0; i < 15; ++i) t.th[i] = th[i];
  t.th[15] = 2.0f;
  bool ok = true;
  for (int s = 0; s < 34; ++s) {
    const double lo = -1.0 + (s - 1) / 16.0, hi = lo + 1.0 / 16.0;
    int base = 0, inside = 0;
    float th_in = 2.0f;
    for (int k = 0; k < 15; ++k) {
      const double v = th[k];
      if (v < lo) {
        ++base;
      } else if (v < hi) {
        ++inside;
        th_in = th[k];
      }
    }
    if (inside > 1) ok = false;
    t.nth[s] = inside ? -th_in : -2.0f;
    t.base1[s] = base + 1;
  }
  t.exact_only = ok ? 0 : 1;
}

template <bool kBf16In, int kR>
static cudaError_t launch_q(const void *W, int64_t nblocks, int group, uint8_t *packed,
                            int8_t *codes, float *absf, float *scale2, int *nonfinite_flag,
                            const QuantTables &tab, int num_sms, cudaStream_t s) {
  constexpr int smem = quant_smem_bytes<kBf16In, kR>();
  static bool set = false;
  if (!set) {
    cudaError_t e = cudaFuncSetAttribute(quantize_nf4_kernel<kBf16In, kR>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    set = true;
  }
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      &per_sm, quantize_nf4_kernel<kBf16In, kR>, quant_launch_threads<kBf16In, kR>(), smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  const int64_t ngroups = (nblocks + 255) / 256;
  int64_t grid = (int64_t)num_sms * per_sm;
  if (grid > ngroups) grid = ngroups;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(quant_launch_threads<kBf16In, kR>(), 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1] = {pdl_attr()};
  cfg.attrs = at;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, quantize_nf4_kernel<kBf16In, kR>, W, nblocks, group, packed, codes,
                         absf, scale2, nonfinite_flag, tab);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_quantize(const void *W, bool bf16_in, int block, int64_t nblocks, int group,
                            uint8_t *packed, int8_t *codes, float *absf, float *scale2,
                            int *nonfinite_flag, const float th[15], int num_sms,
                            cudaStream_t s) {
  if (nblocks == 0) return cudaSuccess;
  QuantTables tab;
  build_quant_tables(th, tab);
  if (block == 64)
    return bf16_in ? launch_q<true, 1>(W, nblocks, group, packed, codes, absf, scale2,
                                       nonfinite_flag, tab, num_sms, s)
                   : launch_q<false, 1>(W, nblocks, group, packed, codes, absf, scale2,
                                        nonfinite_flag, tab, num_sms, s);
  if (block == 128)
    return bf16_in ? launch_q<true, 2>(W, nblocks, group, packed, codes, absf, scale2,
                                       nonfinite_flag, tab, num_sms, s)
                   : launch_q<false, 2>(W, nblocks, group, packed, codes, absf, scale2,
                                        nonfinite_flag, tab, num_sms, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_dequant(const uint8_t *packed, const int8_t *codes, const float *absf,
                           const float *scale2, int group, int block, int64_t nblocks,
                           uint16_t *out, const Codebook &cb, int num_sms, cudaStream_t s) {
  if (nblocks == 0) return cudaSuccess;
  if (block != 64 && block != 128) return cudaErrorInvalidValue;
  const int64_t work = nblocks * (block / 16);
  int64_t grid = (work + 255) / 256;
  const int64_t cap = (int64_t)num_sms * 8 * 4;
  if (grid > cap) grid = cap;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute at[1] = {pdl_attr()};
  cfg.attrs = at;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, dequant_nf4_kernel, packed, codes, absf, scale2, group,
                                     work, block == 64 ? 2 : 3, out, cb);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace qlora
