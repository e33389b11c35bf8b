// capi.cu -- the extern "C" boundary of the QLoRA NF4 library: argument
// validation, workspace layout, TMA descriptor encoding and kernel
// selection.  Every compute step runs in the CUDA kernels of this library.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "kernels.h"


using namespace qlora;

namespace {

// ---------------------------------------------------------------- helpers
inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline int round_up(int v, int m) { return (v + m - 1) / m * m; }
inline size_t round_up_sz(size_t v, size_t m) { return (v + m - 1) / m * m; }

int num_sms_current() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 148;
  return n;
}

// Decision thresholds of the nearest-codepoint rule.  For each pair of
// neighbouring codepoints (c_k, c_{k+1}) the threshold is the smallest fp32 x
// in [c_k, c_{k+1}] whose fp32 distance to c_{k+1} is strictly smaller than
// its fp32 distance to c_k (an exact tie keeps the lower index).  Both
// distances are monotone in x, so a bisection over the ordered fp32 values
// finds it.
uint32_t fkey(float f) {
  uint32_t b;
  std::memcpy(&b, &f, 4);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
float funkey(uint32_t k) {
  const uint32_t b = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
  float f;
  std::memcpy(&f, &b, 4);
  return f;
}
// Percentage points of the normal distribution: Wichura's algorithm AS 241
// (PPND16, Applied Statistics 37(3), 1988), rational approximations with
// about 1e-16 relative accuracy, binary64.
double ppnd16(double p) {
  const double q = p - 0.5;
  if (std::fabs(q) <= 0.425) {
    const double r = 0.180625 - q * q;
    return q *
           (((((((2509.0809287301226727 * r + 33430.575583588128105) * r +
                 67265.770927008700853) * r + 45921.953931549871457) * r +
               13731.693765509461125) * r + 1971.5909503065514427) * r +
             133.14166789178437745) * r + 3.387132872796366608) /
           (((((((5226.495278852854561 * r + 28729.085735721942674) * r +
                 39307.89580009271061) * r + 21213.794301586595867) * r +
               5394.1960214247511077) * r + 687.1870074920579083) * r +
             42.313330701600911252) * r + 1.0);
  }
  double r = q < 0 ? p : 1.0 - p;
  r = std::sqrt(-std::log(r));
  double v;
  if (r <= 5.0) {
    r -= 1.6;
    v = (((((((7.7454501427834140764e-4 * r + 0.0227238449892691845833) * r +
              0.24178072517745061177) * r + 1.27045825245236838258) * r +
            3.64784832476320460504) * r + 5.7694972214606914055) * r +
          4.6303378461565452959) * r + 1.42343711074968357734) /
        (((((((1.05075007164441684324e-9 * r + 5.475938084995344946e-4) * r +
              0.0151986665636164571966) * r + 0.14810397642748007459) * r +
            0.68976733498510000455) * r + 1.6763848301838038494) * r +
          2.05319162663775882187) * r + 1.0);
  } else {
    r -= 5.0;
    v = (((((((2.01033439929228813265e-7 * r + 2.71155556874348757815e-5) * r +
              0.0012426609473880784386) * r + 0.026532189526576123093) * r +
            0.29656057182850489123) * r + 1.7848265399172913358) * r +
          5.4637849111641143699) * r + 6.6579046435011037772) /
        (((((((2.04426310338993978564e-15 * r + 1.4215117583164458887e-7) * r +
              1.8463183175100546818e-5) * r + 7.868691311456132591e-4) * r +
            0.0148753612908506148525) * r + 0.13692988092273580531) * r +
          0.59983220655588793769) * r + 1.0);
  }
  return q < 0 ? -v : v;
}

// The codebooks.  0: the printed NF4 table.  1: the quantile construction
// q_i = Phi^-1((i - 0.5) / 16), i = 1..16 ("QLoRA and 4bit Quantization |
// QLoRA 与 4-bit 量化", Step 2), divided by q_16 so that it runs from -1 to 1;
// the upper half is computed and mirrored (exactly symmetric, no zero).
struct Tables {
  Codebook cb;
  float th[15];
};
Tables g_tab[2];
std::once_flag g_tab_once;

void compute_tables() {
  const float printed[16] = {QLORA_NF4_VALUES};
  for (int i = 0; i < 16; ++i) g_tab[0].cb.v[i] = printed[i];
  const double q16 = ppnd16(15.5 / 16.0);
  for (int i = 9; i <= 16; ++i) {
    const float c = (float)(ppnd16((i - 0.5) / 16.0) / q16);
    g_tab[1].cb.v[i - 1] = c;
    g_tab[1].cb.v[16 - i] = -c;
  }
  for (int t = 0; t < 2; ++t) {
    const float *c = g_tab[t].cb.v;
    for (int k = 0; k < 15; ++k) {
      const float lo = c[k], hi = c[k + 1];
      auto closer_to_hi = [&](float x) {
        volatile float dh = std::fabs(x - hi);
        volatile float dl = std::fabs(x - lo);
        return dh < dl;
      };
      uint32_t a = fkey(lo), b = fkey(hi);  // closer_to_hi(lo) false, (hi) true
      while (b - a > 1) {
        const uint32_t mid = a + (b - a) / 2;
        if (closer_to_hi(funkey(mid)))
          b = mid;
        else
          a = mid;
      }
      g_tab[t].th[k] = funkey(b);
    }
  }
}
const Tables &tables(int codebook) {
  std::call_once(g_tab_once, compute_tables);
  return g_tab[codebook == 1 ? 1 : 0];
}

qlora_status check_weight(const qlora_nf4_weight *w, bool need_buffers) {
  if (!w) return QLORA_ERR_INVALID_ARG;
  if (w->rows < 0 || w->cols < 0) return QLORA_ERR_SHAPE;
  if (w->block != 64 && w->block != 128) return QLORA_ERR_SHAPE;
  if (!(w->group == 0 || w->group == 32 || w->group == 64 || w->group == 128 ||
        w->group == 256))
    return QLORA_ERR_SHAPE;
  if (w->cols % w->block) return QLORA_ERR_SHAPE;
  if (w->codebook != QLORA_CODEBOOK_PRINTED && w->codebook != QLORA_CODEBOOK_QUANTILE)
    return QLORA_ERR_INVALID_ARG;
  if (!need_buffers) return QLORA_OK;
  if (!w->packed) return QLORA_ERR_INVALID_ARG;
  if (w->group > 0 && (!w->absmax_code || !w->scale2)) return QLORA_ERR_INVALID_ARG;
  if (w->group == 0 && !w->absmax_f32) return QLORA_ERR_INVALID_ARG;
  if (!aligned16(w->packed)) return QLORA_ERR_ALIGN;
  if (w->absmax_f32 && (reinterpret_cast<uintptr_t>(w->absmax_f32) & 3u)) return QLORA_ERR_ALIGN;
  if (w->scale2 && (reinterpret_cast<uintptr_t>(w->scale2) & 3u)) return QLORA_ERR_ALIGN;
  return QLORA_OK;
}

// Workspace layout for (M, N, K, r).
// `total_min` is the least a call accepts; `total` adds the split-tile
// area of the fused GEMM (fp32 partial tiles and their counters, sized for
// every cluster the device can run), which calls use when it is there.
struct WsLayout {
  size_t status, t, u, lb, bt, at, part, part_a, gcnt, gcnt_a, total_min, skcnt, skpart, total;
  int sk_clusters;
};
WsLayout ws_layout(int64_t M, int64_t N, int64_t K, int r) {
  const int RP = round_up(r, 16);
  WsLayout L;
  size_t off = 0;
  L.status = off;
  off += 256;
  L.t = off;
  off += round_up_sz((size_t)M * RP * 4, 256);
  L.u = off;
  off += round_up_sz((size_t)M * RP * 4, 256);
  L.lb = off;  // bf16(s.t) or bf16(s.u), [M, RP]: operand of the GEMM's rank-r MMAs
  off += round_up_sz((size_t)M * RP * 2, 256);
  L.bt = off;
  off += round_up_sz((size_t)RP * N * 2, 256);
  L.at = off;
  off += round_up_sz((size_t)K * RP * 2, 256);
  // dB and dA run in one launch: their partial sums and their column-tile
  // counters (zero between calls) are separate, dB's first
  L.part = off;
  int sn = 1, sk = 1;
  skinny_splits_pair(M, (int)N, (int)K, &sn, &sk);
  const size_t pn = (size_t)sn * N, pk = (size_t)sk * K;
  L.part_a = off + round_up_sz(pn * RP * 4, 256);
  off = L.part_a + round_up_sz(pk * RP * 4, 256);
  L.gcnt = off;
  const int tn = skinny_tiles((int)N), tk = skinny_tiles((int)K);
  L.gcnt_a = off + round_up_sz((size_t)tn * sizeof(int), 256);
  off = L.gcnt_a + round_up_sz((size_t)tk * sizeof(int), 256);
  L.total_min = off;
  L.sk_clusters = gemm_cluster_bound();
  L.skcnt = off;
  off += round_up_sz((size_t)L.sk_clusters * 2 * sizeof(int), 256);
  L.skpart = off;
  off += (size_t)L.sk_clusters * 2 * 2 * 128 * 256 * sizeof(float);
  L.total = off;
  return L;
}

// 2-D bf16 tensor map: dims {inner, outer}, row pitch in bytes.
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool make_tmap(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer,
               uint64_t pitch_bytes, uint32_t box_inner, uint32_t box_outer,
               CUtensorMapSwizzle swz,
               CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {pitch_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The down-projection out = G . H^T (G [M, C], H [r, C], bf16 row-major):
// inputs of 8192 columns or more stream through the TMA ring kernel (its two
// tensor maps made here), narrower ones through the register kernel.
cudaError_t run_lora_down(const uint16_t *G, int64_t M, int C, const uint16_t *H, int r, float s,
                          float *out, uint16_t *outb, int r_pad, int *status, cudaStream_t st,
                          const uint32_t *mask = nullptr, int wpr = 0, float keep_scale = 1.0f) {
  if (M == 0) return cudaSuccess;
  if (C < 8192)
    return launch_lora_down(G, M, C, H, r, s, out, outb, r_pad, num_sms_current(), st, mask, wpr,
                            keep_scale);
  const int nt = (r + 7) / 8 + ((r + 7) / 8) % 2;  // an even number of 8-row tiles
  CUtensorMap tmG, tmH;
  if (!make_tmap(&tmG, G, (uint64_t)C, (uint64_t)M, (uint64_t)C * 2, 64, 16,
                 CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap(&tmH, H, (uint64_t)C, (uint64_t)r, (uint64_t)C * 2, 64, (uint32_t)(nt * 8),
                 CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  return launch_lora_down_tma(tmG, tmH, M, C, r, s, out, outb, r_pad, num_sms_current(), status,
                              st, mask, wpr, keep_scale);
}

void set_block_constants(GemmArgs &g, const qlora_nf4_weight *w) {
  g.use_code = w->group > 0;
  g.cvec = w->group > 0 ? w->scale2 : w->absmax_f32;
  g.cdiv = w->group > 0 ? w->group : 1;
  g.cshift = 0;
  while ((1 << g.cshift) < g.cdiv) ++g.cshift;
  g.bshift = w->block == 128 ? 1 : 0;
  g.cb = tables(w->codebook).cb;
  if (!g.use_code) g.codes = reinterpret_cast<const int8_t *>(w->packed);
}

qlora_status cuda_status(cudaError_t e) { return e == cudaSuccess ? QLORA_OK : QLORA_ERR_CUDA; }

void set_gemm_plan(GemmArgs &g, const GemmPlan &plan, const WsLayout &L, uint8_t *wsb) {
  g.sk = plan.sk;
  g.clusters = plan.clusters;
  if (plan.sk) {
    g.sk_count = reinterpret_cast<int *>(wsb + L.skcnt);
    g.sk_part = reinterpret_cast<float *>(wsb + L.skpart);
    g.sk_slots_clusters = L.sk_clusters;
  }
}

qlora_status check_linear_common(const qlora_nf4_weight *w, const uint16_t *x, int64_t M,
                                 const uint16_t *A, const uint16_t *B, int32_t r, void *ws,
                                 size_t ws_bytes) {
  qlora_status st = check_weight(w, true);
  if (st != QLORA_OK) return st;
  if (!x || !A || !B) return QLORA_ERR_INVALID_ARG;
  if (M < 1 || M > (int64_t)INT32_MAX) return QLORA_ERR_SHAPE;
  if (w->rows < 1 || w->cols < kBlock) return QLORA_ERR_SHAPE;
  if (w->rows % 8 || w->rows > (int64_t)INT32_MAX || w->cols > (int64_t)INT32_MAX)
    return QLORA_ERR_SHAPE;
  if (r < 8 || r > 64 || r % 8) return QLORA_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(A) || !aligned16(B)) return QLORA_ERR_ALIGN;
  if (!ws) return QLORA_ERR_WORKSPACE;
  if (!aligned16(ws)) return QLORA_ERR_ALIGN;
  if (ws_bytes < ws_layout(M, w->rows, w->cols, r).total_min) return QLORA_ERR_WORKSPACE;
  return QLORA_OK;
}

}  // namespace

void qlora::ws_counter_range(int64_t M, int64_t N, int64_t K, int r, size_t *off,
                             size_t *bytes) {
  const WsLayout L = ws_layout(M, N, K, r);
  *off = L.gcnt;
  *bytes = L.total_min - L.gcnt;
}

extern "C" {

const char *qlora_status_string(qlora_status s) {
  switch (s) {
    case QLORA_OK: return "ok";
    case QLORA_ERR_INVALID_ARG: return "invalid argument";
    case QLORA_ERR_SHAPE: return "unsupported shape";
    case QLORA_ERR_ALIGN: return "pointer or stride not 16-byte aligned";
    case QLORA_ERR_DTYPE: return "unsupported dtype";
    case QLORA_ERR_NONFINITE: return "non-finite input";
    case QLORA_ERR_TIMEOUT: return "device pipeline wait timed out";
    case QLORA_ERR_CUDA: return "CUDA error";
    case QLORA_ERR_WORKSPACE: return "workspace missing or too small";
  }
  return "unknown status";
}

qlora_status qlora_nf4_codebook(int32_t codebook, float out[16]) {
  if (!out || (codebook != 0 && codebook != 1)) return QLORA_ERR_INVALID_ARG;
  const Tables &t = tables(codebook);
  for (int i = 0; i < 16; ++i) out[i] = t.cb.v[i];
  return QLORA_OK;
}

qlora_status qlora_nf4_thresholds(int32_t codebook, float out[15]) {
  if (!out || (codebook != 0 && codebook != 1)) return QLORA_ERR_INVALID_ARG;
  const Tables &t = tables(codebook);
  for (int i = 0; i < 15; ++i) out[i] = t.th[i];
  return QLORA_OK;
}

qlora_status qlora_nf4_sizes(int64_t rows, int64_t cols, int32_t block, int32_t group,
                             size_t *packed_bytes, size_t *code_bytes, size_t *scale_bytes) {
  if (rows < 0 || cols < 0 || block <= 0 || (block & 1) || group < 0) return QLORA_ERR_SHAPE;
  if (cols % block) return QLORA_ERR_SHAPE;
  const int64_t n = rows * cols, nb = n / block;
  if (packed_bytes) *packed_bytes = (size_t)(n / 2);
  if (code_bytes) *code_bytes = (size_t)(group > 0 ? nb : nb * 4);
  if (scale_bytes) *scale_bytes = (size_t)(group > 0 ? ((nb + group - 1) / group) * 4 : 0);
  return QLORA_OK;
}

qlora_status qlora_quantize_nf4(const void *W, qlora_dtype w_dtype, const qlora_nf4_weight *out,
                                int32_t *nonfinite_flag, void *stream) {
  qlora_status st = check_weight(out, true);
  if (st != QLORA_OK) return st;
  if (!W) return QLORA_ERR_INVALID_ARG;
  if (w_dtype != QLORA_F32 && w_dtype != QLORA_BF16) return QLORA_ERR_DTYPE;
  if (!aligned16(W)) return QLORA_ERR_ALIGN;
  const int64_t nblocks = out->rows * out->cols / out->block;
  return cuda_status(launch_quantize(W, w_dtype == QLORA_BF16, out->block, nblocks, out->group,
                                     out->packed,
                                     out->absmax_code, out->absmax_f32, out->scale2,
                                     nonfinite_flag, tables(out->codebook).th, num_sms_current(),
                                     static_cast<cudaStream_t>(stream)));
}

qlora_status qlora_dequant(const qlora_nf4_weight *w, uint16_t *W_out, void *stream) {
  qlora_status st = check_weight(w, true);
  if (st != QLORA_OK) return st;
  if (!W_out) return QLORA_ERR_INVALID_ARG;
  if (!aligned16(W_out)) return QLORA_ERR_ALIGN;
  const int64_t nblocks = w->rows * w->cols / w->block;
  return cuda_status(launch_dequant(w->packed, w->absmax_code, w->absmax_f32, w->scale2, w->group,
                                    w->block, nblocks, W_out, tables(w->codebook).cb,
                                    num_sms_current(),
                                    static_cast<cudaStream_t>(stream)));
}

qlora_status qlora_merge_lora(const qlora_nf4_weight *w, const uint16_t *A, const uint16_t *B,
                              int32_t r, float alpha, uint16_t *W_out, void *stream) {
  qlora_status st = check_weight(w, true);
  if (st != QLORA_OK) return st;
  if (!A || !B || !W_out) return QLORA_ERR_INVALID_ARG;
  if (r < 8 || r > 64 || r % 8) return QLORA_ERR_SHAPE;
  if (w->rows > (int64_t)INT32_MAX || w->cols > (int64_t)INT32_MAX) return QLORA_ERR_SHAPE;
  if (!aligned16(A) || !aligned16(B) || !aligned16(W_out)) return QLORA_ERR_ALIGN;
  MergeArgs a{};
  a.packed = w->packed;
  a.use_code = w->group > 0;
  a.codes = a.use_code ? w->absmax_code : reinterpret_cast<const int8_t *>(w->packed);
  a.cvec = a.use_code ? w->scale2 : w->absmax_f32;
  const int cdiv = w->group > 0 ? w->group : 1;
  a.cshift = 0;
  while ((1 << a.cshift) < cdiv) ++a.cshift;
  a.bshift = w->block == 128 ? 1 : 0;
  a.N = (int)w->rows;
  a.K = (int)w->cols;
  a.A = A;
  a.B = B;
  a.r = r;
  a.s = alpha / (float)r;
  a.out = W_out;
  a.cb = tables(w->codebook).cb;
  a.k31 = 0x80000000u;
  a.k16 = 0x10000u;
  // W_out as [N][K / 64][64] bf16: one box is a 16-row x 256-column tile
  auto fn = encode_fn();
  if (!fn) return QLORA_ERR_CUDA;
  CUtensorMap tmO;
  const cuuint64_t dims[3] = {64, (cuuint64_t)w->cols / 64, (cuuint64_t)w->rows};
  const cuuint64_t strides[2] = {128, (cuuint64_t)w->cols * 2};
  const cuuint32_t box[3] = {64, 4, 16}, estr[3] = {1, 1, 1};
  if (fn(&tmO, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, W_out, dims, strides, box, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return QLORA_ERR_CUDA;
  return cuda_status(
      launch_merge(tmO, a, num_sms_current(), static_cast<cudaStream_t>(stream)));
}

qlora_status qlora_workspace_size(int64_t M, int64_t N, int64_t K, int32_t r, size_t *bytes) {
  if (!bytes) return QLORA_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 0 || r < 1 || r > 64) return QLORA_ERR_SHAPE;
  *bytes = ws_layout(M, N, K, r).total;
  return QLORA_OK;
}

qlora_status qlora_workspace_size_min(int64_t M, int64_t N, int64_t K, int32_t r, size_t *bytes) {
  if (!bytes) return QLORA_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 0 || r < 1 || r > 64) return QLORA_ERR_SHAPE;
  *bytes = ws_layout(M, N, K, r).total_min;
  return QLORA_OK;
}

qlora_status qlora_workspace_init(void *ws, size_t ws_bytes, void *stream) {
  if (!ws) return QLORA_ERR_INVALID_ARG;
  return cuda_status(cudaMemsetAsync(ws, 0, ws_bytes, static_cast<cudaStream_t>(stream)));
}

qlora_status qlora_device_status(void *ws, int32_t *status, void *stream) {
  if (!ws || !status) return QLORA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, ws, sizeof(v), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess && v != 0) e = cudaMemsetAsync(ws, 0, sizeof(int32_t), s);
  if (e != cudaSuccess) return QLORA_ERR_CUDA;
  *status = v;
  return QLORA_OK;
}

}  // extern "C"

namespace {

int dropout_words(int64_t K) { return (int)((K + 127) / 128 * 4); }

qlora_status check_dropout(const qlora_lora_dropout *dr) {
  if (!dr) return QLORA_OK;
  if (!dr->mask || !(dr->p >= 0.0f && dr->p < 1.0f)) return QLORA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(dr->mask) & 3u) return QLORA_ERR_ALIGN;
  return QLORA_OK;
}

float keep_scale_of(const qlora_lora_dropout *dr) {
  return dr ? (float)(1.0 / (1.0 - (double)dr->p)) : 1.0f;
}

qlora_status linear_fwd_impl(const qlora_nf4_weight *w, const uint16_t *x, int64_t M,
                             const uint16_t *A, const uint16_t *B, int32_t r, float alpha,
                             const qlora_lora_dropout *dr, void *y, qlora_dtype y_dtype,
                             float *t_save, void *ws, size_t ws_bytes, uint32_t flags,
                             void *stream) {
  qlora_status st = check_linear_common(w, x, M, A, B, r, ws, ws_bytes);
  if (st != QLORA_OK) return st;
  st = check_dropout(dr);
  if (st != QLORA_OK) return st;
  const uint32_t *dmask = dr ? dr->mask : nullptr;
  const int dwpr = dropout_words(w->cols);
  const float kscale = keep_scale_of(dr);
  if (!y) return QLORA_ERR_INVALID_ARG;
  if (y_dtype != QLORA_F32 && y_dtype != QLORA_BF16) return QLORA_ERR_DTYPE;
  if (!aligned16(y) || (t_save && !aligned16(t_save))) return QLORA_ERR_ALIGN;
  if ((flags & QLORA_FLAG_FORCE_GEMV) && (flags & QLORA_FLAG_FORCE_GEMM))
    return QLORA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int N = (int)w->rows, K = (int)w->cols;
  const float sc = alpha / (float)r;
  const WsLayout L = ws_layout(M, N, K, r);
  uint8_t *wsb = static_cast<uint8_t *>(ws);
  GemvPlan gplan{};
  const bool gemv_ok = M <= 16 && gemv_plan(N, K, (int)M, r, num_sms_current(), &gplan) == 0;
  const bool use_gemv =
      (flags & QLORA_FLAG_FORCE_GEMV) || (M <= 16 && gemv_ok && !(flags & QLORA_FLAG_FORCE_GEMM));
  if (use_gemv) {
    if (!gemv_ok) return QLORA_ERR_SHAPE;
    CUtensorMap tmW;
    if (!make_tmap(&tmW, w->packed, (uint64_t)K / 2, (uint64_t)N, (uint64_t)K / 2, 128, 16,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_DATA_TYPE_UINT8))
      return QLORA_ERR_CUDA;
    GemvArgs a{};
    a.packed = w->packed;
    a.use_code = w->group > 0;
    a.codes = a.use_code ? w->absmax_code : reinterpret_cast<const int8_t *>(w->packed);
    a.cvec = a.use_code ? w->scale2 : w->absmax_f32;
    const int cdiv = w->group > 0 ? w->group : 1;
    a.cshift = 0;
    while ((1 << a.cshift) < cdiv) ++a.cshift;
    a.bshift = w->block == 128 ? 1 : 0;
    a.N = N;
    a.K = K;
    a.x = x;
    a.M = (int)M;
    a.B = B;
    a.r = r;
    a.RP = round_up(r, 16);
    a.s = sc;
    a.y = y;
    a.y_bf16 = y_dtype == QLORA_BF16;
    a.t = reinterpret_cast<const float *>(wsb + L.t);
    a.status = reinterpret_cast<int *>(wsb + L.status);
    a.cb = tables(w->codebook).cb;
    a.mask = dmask;
    a.wpr = dwpr;
    a.keep_scale = kscale;
    return cuda_status(launch_gemv(tmW, a, gplan, A, reinterpret_cast<float *>(wsb + L.part),
                                   reinterpret_cast<int *>(wsb + L.gcnt), t_save, s));
  }
  const int RP = round_up(r, 16);
  const bool sk_ws = ws_bytes >= L.total;
  GemmPlan plan;
  cudaError_t e = gemm_plan(false, (int)M, N, K, RP, sk_ws ? L.sk_clusters : 0, &plan);
  if (e == cudaErrorInvalidValue) return QLORA_ERR_SHAPE;
  if (e != cudaSuccess) return QLORA_ERR_CUDA;
  const int bn = plan.bn;
  uint16_t *lb = reinterpret_cast<uint16_t *>(wsb + L.lb);
  e = run_lora_down(x, M, K, A, r, sc, t_save, lb, RP, reinterpret_cast<int *>(wsb + L.status), s,
                    dmask, dwpr, kscale);
  if (e != cudaSuccess) return QLORA_ERR_CUDA;
  CUtensorMap tmA, tmL1, tmL2;
  if (!make_tmap(&tmA, x, K, M, (uint64_t)K * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap(&tmL1, lb, RP, M, (uint64_t)RP * 2, 16, 128, CU_TENSOR_MAP_SWIZZLE_32B) ||
      !make_tmap(&tmL2, B, r, N, (uint64_t)r * 2, 16, bn / 2, CU_TENSOR_MAP_SWIZZLE_32B))
    return QLORA_ERR_CUDA;
  GemmArgs g{};
  g.packed = w->packed;
  g.codes = w->absmax_code;
  g.absf = w->absmax_f32;
  g.scale2 = w->scale2;
  g.group = w->group;
  g.wrows = N;
  g.wcols = K;
  g.M = (int)M;
  g.out_cols = N;
  g.kdim = K;
  g.r = r;
  g.r_pad = RP;
  g.s = sc;
  g.out = y;
  g.out_bf16 = y_dtype == QLORA_BF16;
  g.stages = gemm_pick_stages(RP);
  g.status = reinterpret_cast<int *>(wsb + L.status);
  g.bn = bn;
  set_gemm_plan(g, plan, L, wsb);
  set_block_constants(g, w);
  return cuda_status(launch_gemm(false, tmA, tmL1, tmL2, g, s));
}

qlora_status linear_bwd_impl(const qlora_nf4_weight *w, const uint16_t *x, const uint16_t *dY,
                             int64_t M, const uint16_t *A, const uint16_t *B, int32_t r,
                             float alpha, const qlora_lora_dropout *dr, const float *t_saved,
                             void *dX, qlora_dtype dx_dtype, float *dA, float *dB, void *ws,
                             size_t ws_bytes, uint32_t flags, void *stream) {
  (void)flags;
  qlora_status st = check_linear_common(w, x, M, A, B, r, ws, ws_bytes);
  if (st != QLORA_OK) return st;
  st = check_dropout(dr);
  if (st != QLORA_OK) return st;
  if (dr && dx_dtype != QLORA_F32) return QLORA_ERR_DTYPE;
  const uint32_t *dmask = dr ? dr->mask : nullptr;
  const int dwpr = dropout_words(w->cols);
  const float kscale = keep_scale_of(dr);
  if (!dY || !dX || !dA || !dB) return QLORA_ERR_INVALID_ARG;
  if (dx_dtype != QLORA_F32 && dx_dtype != QLORA_BF16) return QLORA_ERR_DTYPE;
  if (!aligned16(dY) || !aligned16(dX) || !aligned16(dA) || !aligned16(dB) ||
      (t_saved && !aligned16(t_saved)))
    return QLORA_ERR_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int N = (int)w->rows, K = (int)w->cols;
  const int RP = round_up(r, 16);
  const float sc = alpha / (float)r;
  const int nsm = num_sms_current();
  const WsLayout L = ws_layout(M, N, K, r);
  uint8_t *wsb = static_cast<uint8_t *>(ws);
  float *u = reinterpret_cast<float *>(wsb + L.u);
  uint16_t *Bt = reinterpret_cast<uint16_t *>(wsb + L.bt);
  uint16_t *At = reinterpret_cast<uint16_t *>(wsb + L.at);
  float *part = reinterpret_cast<float *>(wsb + L.part);
  uint16_t *lb = reinterpret_cast<uint16_t *>(wsb + L.lb);
  const float *t = t_saved;
  cudaError_t e;
  if (!t) {
    float *tw = reinterpret_cast<float *>(wsb + L.t);
    e = run_lora_down(x, M, K, A, r, sc, tw, nullptr, RP, reinterpret_cast<int *>(wsb + L.status),
                      s, dmask, dwpr, kscale);
    if (e != cudaSuccess) return QLORA_ERR_CUDA;
    t = tw;
  }
  e = launch_transposes(A, B, N, K, r, RP, At, Bt, nsm, s);
  if (e != cudaSuccess) return QLORA_ERR_CUDA;
  // u = dY . B (fp32, for dA) and bf16(s . u) (operand of the dX GEMM's rank-r MMAs;
  // with dropout bf16(s / (1 - p) . u), taken back out at the dropped positions)
  e = run_lora_down(dY, M, N, Bt, r, sc * kscale, u, lb, RP,
                    reinterpret_cast<int *>(wsb + L.status), s);
  if (e != cudaSuccess) return QLORA_ERR_CUDA;
  GemmPlan plan;
  e = gemm_plan(true, (int)M, K, N, RP, ws_bytes >= L.total ? L.sk_clusters : 0, &plan);
  if (e == cudaErrorInvalidValue) return QLORA_ERR_SHAPE;
  if (e != cudaSuccess) return QLORA_ERR_CUDA;
  const int bn = plan.bn;
  CUtensorMap tmA, tmL1, tmL2;
  if (!make_tmap(&tmA, dY, N, M, (uint64_t)N * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap(&tmL1, lb, RP, M, (uint64_t)RP * 2, 16, 128, CU_TENSOR_MAP_SWIZZLE_32B) ||
      !make_tmap(&tmL2, At, RP, K, (uint64_t)RP * 2, 16, bn / 2, CU_TENSOR_MAP_SWIZZLE_32B))
    return QLORA_ERR_CUDA;
  GemmArgs g{};
  g.packed = w->packed;
  g.codes = w->absmax_code;
  g.absf = w->absmax_f32;
  g.scale2 = w->scale2;
  g.group = w->group;
  g.wrows = N;
  g.wcols = K;
  g.M = (int)M;
  g.out_cols = K;
  g.kdim = N;
  g.r = r;
  g.r_pad = RP;
  g.s = sc;
  g.out = dX;
  g.out_bf16 = dx_dtype == QLORA_BF16;
  g.stages = gemm_pick_stages(RP);
  g.status = reinterpret_cast<int *>(wsb + L.status);
  g.bn = bn;
  set_gemm_plan(g, plan, L, wsb);
  set_block_constants(g, w);
  e = launch_gemm(true, tmA, tmL1, tmL2, g, s);
  if (e != cudaSuccess) return QLORA_ERR_CUDA;
  if (dmask) {
    e = launch_dropout_dx_fix(dmask, dwpr, M, K, lb, At, RP, static_cast<float *>(dX), nsm, s);
    if (e != cudaSuccess) return QLORA_ERR_CUDA;
  }
  // dB = s . dY^T . t and dA = s . u^T . x (with dropout s / (1 - p) . u^T . (x . keep)),
  // one launch
  int *gcnt = reinterpret_cast<int *>(wsb + L.gcnt);
  int *gcnt_a = reinterpret_cast<int *>(wsb + L.gcnt_a);
  float *part_a = reinterpret_cast<float *>(wsb + L.part_a);
  int sn = 1, sk = 1;
  skinny_splits_pair(M, N, K, &sn, &sk);
  const SkinnyJob jb = skinny_job(dY, M, N, t, part, gcnt, sn, sc, false, dB, nullptr, 0);
  const SkinnyJob ja = skinny_job(x, M, K, u, part_a, gcnt_a, sk, sc * kscale, true, dA, dmask,
                                  dwpr);
  e = launch_skinny2(jb, ja, M, r, RP, s);
  return cuda_status(e);
}

}  // namespace

extern "C" {

qlora_status qlora_linear_fwd(const qlora_nf4_weight *w, const uint16_t *x, int64_t M,
                              const uint16_t *A, const uint16_t *B, int32_t r, float alpha,
                              void *y, qlora_dtype y_dtype, float *t_save, void *ws,
                              size_t ws_bytes, uint32_t flags, void *stream) {
  return linear_fwd_impl(w, x, M, A, B, r, alpha, nullptr, y, y_dtype, t_save, ws, ws_bytes,
                         flags, stream);
}

qlora_status qlora_linear_fwd_dropout(const qlora_nf4_weight *w, const uint16_t *x, int64_t M,
                                      const uint16_t *A, const uint16_t *B, int32_t r,
                                      float alpha, const qlora_lora_dropout *dropout, void *y,
                                      qlora_dtype y_dtype, float *t_save, void *ws,
                                      size_t ws_bytes, uint32_t flags, void *stream) {
  if (!dropout) return QLORA_ERR_INVALID_ARG;
  return linear_fwd_impl(w, x, M, A, B, r, alpha, dropout, y, y_dtype, t_save, ws, ws_bytes,
                         flags, stream);
}

qlora_status qlora_linear_bwd(const qlora_nf4_weight *w, const uint16_t *x, const uint16_t *dY,
                              int64_t M, const uint16_t *A, const uint16_t *B, int32_t r,
                              float alpha, const float *t_saved, void *dX, qlora_dtype dx_dtype,
                              float *dA, float *dB, void *ws, size_t ws_bytes, uint32_t flags,
                              void *stream) {
  return linear_bwd_impl(w, x, dY, M, A, B, r, alpha, nullptr, t_saved, dX, dx_dtype, dA, dB, ws,
                         ws_bytes, flags, stream);
}

qlora_status qlora_linear_bwd_dropout(const qlora_nf4_weight *w, const uint16_t *x,
                                      const uint16_t *dY, int64_t M, const uint16_t *A,
                                      const uint16_t *B, int32_t r, float alpha,
                                      const qlora_lora_dropout *dropout, const float *t_saved,
                                      float *dX, float *dA, float *dB, void *ws, size_t ws_bytes,
                                      uint32_t flags, void *stream) {
  if (!dropout) return QLORA_ERR_INVALID_ARG;
  return linear_bwd_impl(w, x, dY, M, A, B, r, alpha, dropout, t_saved, dX, QLORA_F32, dA, dB,
                         ws, ws_bytes, flags, stream);
}

qlora_status qlora_dropout_mask_words(int64_t K, int64_t *words_per_row) {
  if (!words_per_row || K < 0) return QLORA_ERR_INVALID_ARG;
  *words_per_row = dropout_words(K);
  return QLORA_OK;
}

qlora_status qlora_dropout_mask(uint64_t seed, float p, int64_t M, int64_t K, uint32_t *mask,
                                void *stream) {
  if (!mask || !(p >= 0.0f && p < 1.0f) || M < 0 || K < 0) return QLORA_ERR_INVALID_ARG;
  if (K % 64 || K > (int64_t)INT32_MAX) return QLORA_ERR_SHAPE;
  if (reinterpret_cast<uintptr_t>(mask) & 15u) return QLORA_ERR_ALIGN;
  double t = std::floor((double)p * 4294967296.0 + 0.5);
  if (t > 4294967295.0) t = 4294967295.0;
  return cuda_status(launch_dropout_mask(seed, (uint32_t)t, M, (int)K, dropout_words(K), mask,
                                         num_sms_current(), static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
