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
// Both kernels are HBM-bound.  Layout of the work:
//   quantise: one CTA of 256 threads per 256 consecutive blocks (one double
//     quantisation group of 256, or several smaller groups).  Eight lanes
//     share a block: each lane reads 16 bytes of bf16 (or 32 of fp32), the
//     block maximum is an 8-lane shuffle reduction, and the lane writes its
//     8 indices as one 32-bit word, so each warp instruction moves 512
//     contiguous bytes in and 128 contiguous bytes out.  All eight passes of
//     a thread are loaded before the first is used.
//   dequantise: four lanes per block, 16 elements per lane; the per-block
//     scaled table T[i] = bf16(c_i * a_hat) is built once per lane and
//     indexed with byte permutes (the same routine the fused GEMM producer
//     uses), 32-byte stores.
#include "common.cuh"
#include "kernels.h"

namespace qlora {

struct Thresholds {
  float th[16];  // 15 used: index = #{k : x >= th[k]}
};

// Number of thresholds <= x, by bisection over the sorted thresholds.
__device__ __forceinline__ int nf4_index(float x, const float *th) {
  int i = (x >= th[7]) ? 8 : 0;
  i += (x >= th[i + 3]) ? 4 : 0;
  i += (x >= th[i + 1]) ? 2 : 0;
  i += (x >= th[i]) ? 1 : 0;
  return i;
}

template <bool kBf16In>
__global__ void __launch_bounds__(256) quantize_nf4_kernel(const void *__restrict__ W,
                                                           int64_t nblocks, int group,
                                                           uint8_t *__restrict__ packed,
                                                           int8_t *__restrict__ codes,
                                                           float *__restrict__ absf,
                                                           float *__restrict__ scale2,
                                                           int *__restrict__ nonfinite_flag,
                                                           Thresholds thr) {
  __shared__ float th_s[16];
  __shared__ float amax_s[256];
  __shared__ float wmax_s[8];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int sub = lane >> 3, li = lane & 7;
  if (tid == 0) {
#pragma unroll
    for (int i = 0; i < 16; ++i) th_s[i] = thr.th[i];
  }

  const int64_t blk0 = (int64_t)blockIdx.x * 256;

  // Issue every load of this thread first (8 passes x 8 elements).
  float v[8][8];
  bool inb[8];
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    const int b = p * 32 + warp * 4 + sub;
    const int64_t gb = blk0 + b;
    inb[p] = gb < nblocks;
    if (kBf16In) {
      uint4 u = make_uint4(0, 0, 0, 0);
      if (inb[p])
        u = ldg_nc_v4(reinterpret_cast<const uint16_t *>(W) + gb * kBlock + li * 8);
      const uint32_t ww[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        v[p][2 * e] = bf16_lo(ww[e]);
        v[p][2 * e + 1] = bf16_hi(ww[e]);
      }
    } else {
      uint4 u0 = make_uint4(0, 0, 0, 0), u1 = u0;
      if (inb[p]) {
        const float *src = reinterpret_cast<const float *>(W) + gb * kBlock + li * 8;
        u0 = ldg_nc_v4(src);
        u1 = ldg_nc_v4(src + 4);
      }
      v[p][0] = __uint_as_float(u0.x), v[p][1] = __uint_as_float(u0.y);
      v[p][2] = __uint_as_float(u0.z), v[p][3] = __uint_as_float(u0.w);
      v[p][4] = __uint_as_float(u1.x), v[p][5] = __uint_as_float(u1.y);
      v[p][6] = __uint_as_float(u1.z), v[p][7] = __uint_as_float(u1.w);
    }
  }
  __syncthreads();  // th_s visible

  int nonfinite = 0;
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    const int b = p * 32 + warp * 4 + sub;
    float amax = 0.0f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float x = v[p][e];
      if (isfinite(x)) {
        amax = fmaxf(amax, fabsf(x));
      } else {
        ++nonfinite;
      }
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
    if (li == 0) amax_s[b] = amax;  // 0 for blocks past the end
    uint32_t word = 0;
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      int q0 = kZeroIndex, q1 = kZeroIndex;
      if (amax != 0.0f) {
        q0 = nf4_index(__fdiv_rn(v[p][e], amax), th_s);
        q1 = nf4_index(__fdiv_rn(v[p][e + 1], amax), th_s);
      }
      word |= (uint32_t)((q0 << 4) | q1) << (4 * e);  // byte e/2
    }
    if (inb[p]) {
      const int64_t gb = blk0 + b;
      *reinterpret_cast<uint32_t *>(packed + gb * (kBlock / 2) + li * 4) = word;
    }
  }
  if (nonfinite_flag) {
    nonfinite = __any_sync(0xffffffffu, nonfinite != 0);
    if (nonfinite && lane == 0) atomicExch(nonfinite_flag, 1);
  }
  __syncthreads();

  // Second level: one scale per `group` consecutive block constants.
  const float a = amax_s[tid];
  const int64_t gb = blk0 + tid;
  if (group == 0) {
    if (gb < nblocks) absf[gb] = a;
    return;
  }
  float m = a;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) wmax_s[warp] = m;
  __syncthreads();
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

// ------------------------------------------------------------- dequantise
__global__ void __launch_bounds__(256) dequant_nf4_kernel(const uint8_t *__restrict__ packed,
                                                          const int8_t *__restrict__ codes,
                                                          const float *__restrict__ absf,
                                                          const float *__restrict__ scale2,
                                                          int group, int64_t nblocks,
                                                          uint16_t *__restrict__ out) {
  const int64_t nquads = nblocks * 4;  // 16-element pieces
  for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < nquads;
       q += (int64_t)gridDim.x * blockDim.x) {
    const int64_t b = q >> 2;
    const uint2 pk = ldg_nc_v2(packed + q * 8);
    float ahat;
    if (group > 0)
      ahat = __fmul_rn((float)codes[b], scale2[b / group]);
    else
      ahat = absf[b];
    const Nf4Table t = make_table(ahat);
    uint32_t o[8];
    lookup8(t, pk.x, o);
    lookup8(t, pk.y, o + 4);
    uint4 *dst = reinterpret_cast<uint4 *>(out + q * 16);
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

// ----------------------------------------------------------- host launchers
cudaError_t launch_quantize(const void *W, bool bf16_in, int64_t nblocks, int group,
                            uint8_t *packed, int8_t *codes, float *absf, float *scale2,
                            int *nonfinite_flag, const float th[15], cudaStream_t s) {
  if (nblocks == 0) return cudaSuccess;
  Thresholds thr;
  for (int i = 0; i < 15; ++i) thr.th[i] = th[i];
  thr.th[15] = 2.0f;
  const int64_t grid = (nblocks + 255) / 256;
  if (bf16_in)
    quantize_nf4_kernel<true><<<(unsigned)grid, 256, 0, s>>>(W, nblocks, group, packed, codes,
                                                             absf, scale2, nonfinite_flag, thr);
  else
    quantize_nf4_kernel<false><<<(unsigned)grid, 256, 0, s>>>(W, nblocks, group, packed, codes,
                                                              absf, scale2, nonfinite_flag, thr);
  return cudaGetLastError();
}

cudaError_t launch_dequant(const uint8_t *packed, const int8_t *codes, const float *absf,
                           const float *scale2, int group, int64_t nblocks, uint16_t *out,
                           int num_sms, cudaStream_t s) {
  if (nblocks == 0) return cudaSuccess;
  const int64_t work = nblocks * 4;
  int64_t grid = (work + 255) / 256;
  const int64_t cap = (int64_t)num_sms * 8 * 4;
  if (grid > cap) grid = cap;
  dequant_nf4_kernel<<<(unsigned)grid, 256, 0, s>>>(packed, codes, absf, scale2, group, nblocks,
                                                    out);
  return cudaGetLastError();
}

}  // namespace qlora
