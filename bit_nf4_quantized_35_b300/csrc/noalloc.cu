// noalloc.cu -- a backward entry point for callers that cannot allocate
// device memory.
//
// qlora_linear_bwd needs a caller-provided workspace (the u = dY.B factor,
// transposed copies of the LoRA matrices and the partial sums of the dA/dB
// reductions).  Some callers cannot call cudaMalloc: code running while a
// CUDA graph is being captured, allocators that forbid allocation on a hot
// path, or hosts that hand the library only its inputs and outputs.  For
// them qlora_linear_bwd_noalloc takes its workspace from a fixed array in
// the library's own device memory, QLORA_NOALLOC_SCRATCH_BYTES long, which
// every GPU that loads the library holds until the process exits.
#include <mutex>

#include "common.cuh"
#include "kernels.h"


namespace {

// The workspace of every qlora_linear_bwd_noalloc call on this device.
// Host code must not pass this symbol to a kernel: in host code it names a
// host-side stand-in; the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) uint8_t g_noalloc_scratch[QLORA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (with that device current) and cached.
qlora_status scratch_address(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QLORA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return QLORA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return QLORA_OK;
}

}  // namespace

extern "C" qlora_status qlora_linear_bwd_noalloc(const qlora_nf4_weight *w, const uint16_t *x,
                                                 const uint16_t *dY, int64_t M,
                                                 const uint16_t *A, const uint16_t *B, int32_t r,
                                                 float alpha, const float *t_saved, void *dX,
                                                 qlora_dtype dx_dtype, float *dA, float *dB,
                                                 uint32_t flags, void *stream) {
  if (!w) return QLORA_ERR_INVALID_ARG;
  size_t need = 0;
  qlora_status st = qlora_workspace_size_min(M, w->rows, w->cols, r, &need);
  if (st != QLORA_OK) return st;
  if (need > (size_t)QLORA_NOALLOC_SCRATCH_BYTES) return QLORA_ERR_WORKSPACE;
  void *ws = nullptr;
  st = scratch_address(&ws);
  if (st != QLORA_OK) return st;
  // Two parts of the workspace are read before this call writes them: the
  // device status word (first 256 bytes) and the dA/dB column-tile counters,
  // which must start at zero.  The counters' place depends on the sizes, so
  // an earlier call of other sizes (or one that timed out) may have left
  // other data there.  Both are zeroed on the caller's stream first; every
  // other byte the backward reads it has written itself.
  size_t cnt_off = 0, cnt_bytes = 0;
  qlora::ws_counter_range(M, w->rows, w->cols, r, &cnt_off, &cnt_bytes);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t *wsb = static_cast<uint8_t *>(ws);
  if (cudaMemsetAsync(wsb, 0, 256, s) != cudaSuccess ||
      cudaMemsetAsync(wsb + cnt_off, 0, cnt_bytes, s) != cudaSuccess)
    return QLORA_ERR_CUDA;
  // `need` bytes (no split-tile area): the dX GEMM computes whole tiles.
  return qlora_linear_bwd(w, x, dY, M, A, B, r, alpha, t_saved, dX, dx_dtype, dA, dB, ws, need,
                          flags, stream);
}
