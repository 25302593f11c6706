// Output stage for callers that cannot allocate device memory.
//
// mtp_head_logits_argmax_batched needs a small device workspace (a completion counter, each
// sequence's running pick and the norm parts of the batched sweep). Some callers cannot provide
// one: a plug-in that
// only ever receives the buffers its host framework hands it and has no allocator of its own,
// or a process whose device memory has all been claimed up front by another allocator. For them
// this file keeps that workspace in a fixed device array owned by the library (the same size
// for every batch the output stage accepts) and runs the unchanged output-stage kernels on it.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/mtp_head.h"
#include "common.cuh"
#include "internal.h"

namespace {

// The output stage's workspace (2304 bytes, the same for every batch size).
constexpr size_t kStaticScratchBytes = static_cast<size_t>(mtp::kWsBytes);

// Every GPU that loads the library holds this array until the process exits. It is zero at load
// time; each output-stage kernel returns its counter to zero, and each call clears it again
// before launching.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once per device. In
// host code the array's name is only a stand-in; the kernels need this address.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (err != cudaSuccess) return err;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" int mtp_head_logits_argmax_batched_noalloc(const uint16_t* x, const uint16_t* final_norm_w,
                                                      const void* lm_head, const float* row_scale,
                                                      int w_dtype, float* logits, int32_t* draft,
                                                      int32_t* status, int B, int H, int V, float eps,
                                                      void* stream) {
  // the scratch holds the workspace of any batch the output stage takes; others are refused
  if (B < 1 || B > mtp::kMaxB) return MTP_ERR_SHAPE;
  if (mtp::sweep_workspace_bytes(B) > kStaticScratchBytes) return MTP_ERR_WORKSPACE;
  void* ws = nullptr;
  if (scratch_address(&ws) != cudaSuccess) return MTP_ERR_CUDA;
  const int v = mtp::check_output_args(x, final_norm_w, lm_head, row_scale, w_dtype, logits, draft,
                                       status, ws, kStaticScratchBytes, B, H, V, eps);
  if (v != MTP_OK) return v;
  // the completion counter and the running picks must start at zero
  if (cudaMemsetAsync(ws, 0, mtp::kWsBytes, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MTP_ERR_CUDA;
  return mtp_head_logits_argmax_batched(x, final_norm_w, lm_head, row_scale, w_dtype, logits, draft,
                                        status, ws, kStaticScratchBytes, B, H, V, eps, stream);
}
