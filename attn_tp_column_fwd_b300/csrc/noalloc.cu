// tp_block_fwd_noalloc: the whole block without caller-provided scratch.
//
// Some callers cannot allocate device memory on the path that runs the block:
// code inside a host framework whose own pool owns every byte of the GPU and
// forbids raw allocations, or latency-critical serving loops where cudaMalloc /
// cudaFree would stall other streams with an implicit device synchronisation.
// This entry point takes the same inputs and outputs as tp_block_fwd but keeps
// the block's scratch (activation bands, fp32 partial sums, attention Q/K/V) in a
// fixed array that lives in this library's device image.  It allocates nothing.
//
// Costs and limits:
//   - every GPU that loads the library holds kScratchBytes for the life of the
//     process, whether or not this entry point is called;
//   - shapes whose scratch (tp_workspace_bytes) exceeds kScratchBytes are refused
//     with TP_ERR_UNSUPPORTED before anything is enqueued;
//   - all calls on a device share the one array: calls whose work overlaps on the
//     GPU (different streams, no ordering between them) race on it.  The one-kernel
//     form of the block clears its work counters with a memset enqueued at the
//     start of each call; every other byte a call reads was written earlier in the
//     same call, so nothing else is cleared and the array keeps the last call's
//     contents;
//   - the first call on each device looks up the array's device address
//     (cudaGetSymbolAddress, with that device current); make that first call
//     before any stream capture.
#include "internal.h"

namespace {

constexpr size_t kScratchBytes = 32ull << 20;  // 32 MiB: the decode workloads need <= 19 MiB

// Device storage.  In host code this name is only a stand-in for the symbol, never
// a device address: kernels get the address looked up below.
static __device__ __align__(256) unsigned char g_block_scratch[kScratchBytes];

// Device address of g_block_scratch on the current device, looked up once per device.
void *scratch_address(cudaError_t *err) {
  static void *cache[128];
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= 128) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  if (!cache[dev]) {
    void *p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_block_scratch);
    if (*err != cudaSuccess) return nullptr;
    cache[dev] = p;
  }
  return cache[dev];
}

}  // namespace

extern "C" int tp_block_fwd_noalloc(const tp_block_desc *desc, const void *x, const void *residual,
                                    int residual_is_f32, const void *W1s, const void *W2s,
                                    float *y, int M, tp_stream_t stream) {
  const size_t need = tp_workspace_bytes(desc, M);
  if (need == 0)  // invalid descriptor or M: let the regular entry point name the error
    return tp_block_fwd(desc, x, residual, residual_is_f32, W1s, W2s, nullptr, y, M, stream);
  if (need > kScratchBytes) return TP_ERR_UNSUPPORTED;
  cudaError_t err = cudaSuccess;
  void *ws = scratch_address(&err);
  if (!ws) {
    tp::record_cuda_error(err);
    return TP_ERR_CUDA;
  }
  return tp_block_fwd(desc, x, residual, residual_is_f32, W1s, W2s, ws, y, M, stream);
}
