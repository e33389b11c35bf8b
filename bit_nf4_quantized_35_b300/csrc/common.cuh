// common.cuh -- small device helpers shared by the QLoRA NF4 kernels:
// the NF4 table, bf16 packing, mbarrier / TMA / tcgen05 inline PTX.
// Written for sm_103a (B300).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "qlora.h"

namespace qlora {

// The 16 NF4 codepoints ("QLoRA and 4bit Quantization | QLoRA 与 4-bit 量化",
// Step 4, create_nf4_lookup_table): each entry is the fp32 value nearest to
// the printed decimal.  Index 7 is the exact zero.
#define QLORA_NF4_VALUES                                                             \
  -1.0f, -0.696f, -0.525f, -0.395f, -0.284f, -0.185f, -0.091f, 0.0f, 0.080f, 0.161f, \
      0.246f, 0.338f, 0.441f, 0.563f, 0.723f, 1.0f

constexpr int kBlock = 64;          // weights per absmax block
constexpr int kZeroIndex = 7;       // index of the exact-zero codepoint

__device__ __forceinline__ float nf4_value(int i) {
  // Compile-time selection; used where the index is a loop constant.
  constexpr float v[16] = {QLORA_NF4_VALUES};
  return v[i];
}

// Device status word values (the first int32 of a workspace).
constexpr int kStatusTimeout = QLORA_ERR_TIMEOUT;

// ---------------------------------------------------------------- bit helpers
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Two fp32 -> one bf16x2 word, round to nearest even; `lo` lands in bits 0-15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------ NF4 block table
// Scaled per-block table in bf16: T[i] = bf16_rn(codepoint[i] * a_hat).  It
// is held as byte planes so that a nibble can index it with `prmt`:
//   lo[q] holds the low bytes of T[4q..4q+3], hi[q] the high bytes.
struct Nf4Table {
  uint32_t lo[4];
  uint32_t hi[4];
};

// The 16 codepoints a kernel dequantises with, passed by value in its
// parameters (the printed table, or the quantile-formula table): the
// products below read them from the constant bank.
struct Codebook {
  float v[16];
};

__device__ __forceinline__ Nf4Table make_table(float ahat, const Codebook &cb) {
  uint32_t P[8];
#pragma unroll
  for (int j = 0; j < 8; ++j)
    P[j] = pack_bf16x2(__fmul_rn(cb.v[2 * j], ahat), __fmul_rn(cb.v[2 * j + 1], ahat));
  Nf4Table t;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    t.lo[q] = prmt(P[2 * q], P[2 * q + 1], 0x6420u);
    t.hi[q] = prmt(P[2 * q], P[2 * q + 1], 0x7531u);
  }
  return t;
}

// Dequantise the 8 indices of one packed 32-bit word (byte j holds elements
// 2j [high nibble] and 2j+1 [low nibble]) to 8 bf16 values, element e in
// half (e & 1) of out[e >> 1].  m = w & 0x77777777 holds the low 3 bits of
// each index, s = ((w >> 1) & 0x44444444) | 0x32103210 chooses the byte by
// bit 3; m_hi and s_hi are m >> 16 and s >> 16.
__device__ __forceinline__ void lookup8_parts(const Nf4Table &t, uint32_t m, uint32_t s,
                                              uint32_t m_hi, uint32_t s_hi, uint32_t out[4]) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t mh = h ? m_hi : m;
    const uint32_t sh = h ? s_hi : s;
    const uint32_t la = prmt(t.lo[0], t.lo[1], mh);
    const uint32_t lb = prmt(t.lo[2], t.lo[3], mh);
    const uint32_t ha = prmt(t.hi[0], t.hi[1], mh);
    const uint32_t hb = prmt(t.hi[2], t.hi[3], mh);
    const uint32_t lo = prmt(la, lb, sh);
    const uint32_t hi = prmt(ha, hb, sh);
    // nibble order inside the 16-bit half is (e1, e0, e3, e2)
    out[2 * h + 0] = prmt(lo, hi, 0x4051u);
    out[2 * h + 1] = prmt(lo, hi, 0x6273u);
  }
}
__device__ __forceinline__ void lookup8(const Nf4Table &t, uint32_t w, uint32_t out[4]) {
  const uint32_t m = w & 0x77777777u;
  const uint32_t s = ((w >> 1) & 0x44444444u) | 0x32103210u;
  lookup8_parts(t, m, s, m >> 16, s >> 16, out);
}
// The same with the three right shifts done as high-word multiplies by
// k31 = 2^31 and k16 = 2^16 (kernel parameters, so that the compiler cannot
// turn them back into shifts): they then run on the multiply pipe instead of
// the integer pipe that carries the byte permutes.
__device__ __forceinline__ uint32_t mul_hi_u32(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.hi.u32 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ void lookup8_mulhi(const Nf4Table &t, uint32_t w, uint32_t out[4],
                                              uint32_t k31, uint32_t k16) {
  const uint32_t m = w & 0x77777777u;
  const uint32_t s = (mul_hi_u32(w, k31) & 0x44444444u) | 0x32103210u;
  lookup8_parts(t, m, s, mul_hi_u32(m, k16), mul_hi_u32(s, k16), out);
}

// Bit mask of 8 bf16 elements (bits of `byte`, element e = bit e) as four
// AND masks of bf16 pairs (element 2p in the low half of word p).
__device__ __forceinline__ void keep_masks(uint32_t byte, uint32_t (&mk)[4]) {
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const uint32_t b = byte >> (2 * p);
    mk[p] = ((b & 1u) ? 0x0000ffffu : 0u) | ((b & 2u) ? 0xffff0000u : 0u);
  }
}

// ------------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Shared-memory error flag of a CTA, accessed with explicit shared-space
// instructions (a generic access would queue behind in-flight global loads).
__device__ __forceinline__ uint32_t ld_shared_volatile(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.volatile.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void st_shared_volatile(uint32_t addr, uint32_t v) {
  asm volatile("st.volatile.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// Bounded wait: tries the barrier first (the common, fast case touches
// nothing else); otherwise spins for at most ~2 s of SM cycles, then
// records QLORA_ERR_TIMEOUT in the device status word and in the CTA's
// shared error flag (at shared address `err`) and returns false.  Once the
// flag is set every later wait that would block returns false at once, so
// all roles run to the end of the kernel.
template <bool kCluster>
__device__ __forceinline__ bool mbar_wait_bounded_t(uint32_t bar, uint32_t parity, uint32_t err,
                                                    int *status) {
  auto try_once = [&]() {
    return kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
  };
  if (try_once()) return true;
  if (ld_shared_volatile(err)) return false;
  const long long t0 = clock64();
  uint32_t n = 0;
  while (!try_once()) {
    if ((++n & 255u) == 0) {
      if (ld_shared_volatile(err)) return false;
      if (clock64() - t0 > (1ll << 32)) {  // ~2 s at 2 GHz
        st_shared_volatile(err, 1u);
        if (status) atomicExch(status, kStatusTimeout);
        return false;
      }
    }
  }
  return true;
}
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint32_t err,
                                                  int *status) {
  return mbar_wait_bounded_t<false>(bar, parity, err, status);
}
__device__ __forceinline__ bool mbar_wait_bounded_cluster(uint32_t bar, uint32_t parity,
                                                          uint32_t err, int *status) {
  return mbar_wait_bounded_t<true>(bar, parity, err, status);
}

// Bounded drain used only on the error path: waits for a phase regardless
// of the CTA error flag, for at most ~0.1 s.
__device__ __forceinline__ void mbar_drain(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > (1ll << 28)) return;
  }
}

// ------------------------------------------------------------------------ TMA
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int32_t c0, int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// -------------------------------------------------------------------- tcgen05
// Shared-memory matrix descriptor (tcgen05 "matrix descriptor"):
//   bits  0-13 start address >> 4
//   bits 16-29 leading-dimension byte offset >> 4
//   bits 32-45 stride-dimension byte offset >> 4
//   bits 46-47 descriptor version (1)
//   bits 49-51 base offset (0: every operand tile here is pattern-aligned)
//   bits 61-63 swizzle: 0 none, 2 128-byte, 4 64-byte, 6 32-byte
__device__ __forceinline__ uint64_t make_sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                               uint32_t swz) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3fffu);
  d |= (uint64_t)((lbo >> 4) & 0x3fffu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3fffu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)(swz & 7u) << 61;
  return d;
}
constexpr uint32_t kSwz128 = 2, kSwz32 = 6;

// Instruction descriptor, kind::f16 with bf16 A/B and fp32 D:
//   bits 4-5 D format (1 = f32), 7-9 A format (1 = bf16), 10-12 B format,
//   bit 15 A major (0 = K), bit 16 B major (1 = MN), 17-22 N >> 3, 24-28 M >> 4
__host__ __device__ constexpr uint32_t make_idesc_bf16(int M, int N, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// cta_group::2 forms: one leader thread drives the tensor cores of a CTA
// pair; completions are multicast to the same barrier offset in both CTAs.
__device__ __forceinline__ void tc_mma2(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Warp-wide forms: every lane of a converged warp executes the call with the
// same operands and one elected lane issues the instruction, so the warp's
// control flow stays uniform (its operands can live in uniform registers).
__device__ __forceinline__ void tc_mma2_elect(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void tc_commit2_mc_elect(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;\n\t}" ::"r"(bar),
      "h"(cta_mask)
      : "memory");
}
__device__ __forceinline__ void tc_commit2_mc(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(cta_mask)
      : "memory");
}
__device__ __forceinline__ void tmem_alloc2(uint32_t slot_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   slot_smem),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc2(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// ---------------------------------------------------------------- cluster
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
// Shared::cluster address of the same shared-memory offset in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
// Arrive on a barrier of another CTA of the cluster (default semantics; a
// cluster-scope release here costs a fence per arrive).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   slot_smem),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// 32 lanes x 32 consecutive fp32 columns: thread i of the warp gets lane
// (base lane + i), columns [col, col + 32).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
        "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]),
        "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
        "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]),
        "=r"(v[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
        "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ------------------------------------------------------------ global loads
__device__ __forceinline__ uint4 ldg_nc_v4(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint2 ldg_nc_v2(const void *p) {
  uint2 v;
  asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}
// Scalar read-only loads kept in program order (asm volatile): a prefetch
// issued early must not be sunk by the compiler to the point of use.
__device__ __forceinline__ int ldg_nc_s8(const int8_t *p) {
  int v;
  asm volatile("ld.global.nc.s8 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ float ldg_nc_f32(const float *p) {
  float v;
  asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ void sts_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                       uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}
// 16-byte global -> shared copy (cp.async); bytes past src_bytes are zero-filled.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// Programmatic dependent launch.  A kernel launched with the attribute may
// start while the kernel before it on the stream is finishing; it does only
// on-chip set-up before pdl_wait_release(), which waits until that kernel has
// completed and its writes are visible, so every global read and write after
// it keeps stream order.  The release lets the next kernel start the same way.
__device__ __forceinline__ void pdl_wait_release() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
inline cudaLaunchAttribute pdl_attr() {
  cudaLaunchAttribute a;
  a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a.val.programmaticStreamSerializationAllowed = 1;
  return a;
}

__device__ __forceinline__ uint4 lds_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

}  // namespace qlora
