// Host <-> device moves of the host-buffer draft step as kernels, for its recorded CUDA graph:
// the inputs are read straight from mapped pinned host memory (zero copy) and the draft written
// straight back (for one sequence by the sweep's last CTA itself, host_back.h; otherwise by
// host_out_kernel after the sweep). Against the three copy operations they replace (~13 us of GPU time a step),
// they need no copy engine, and with programmatic dependent launch the input stage starts its
// weight stream while the first one runs and the last one is waiting for the sweep.
// Plain loads and stores only: a host-mapped address is a valid global address for them.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

namespace mtp {

namespace {

constexpr int kIoThreads = 256;
constexpr int kIoPer = 4;  // 16-byte pieces a thread has in flight at once (host memory is far away)

// Grid: ceil(n16 / (kIoThreads * kIoPer)) CTAs; CTA 0 also moves the tokens (B <= 16).
__global__ void __launch_bounds__(kIoThreads) host_in_kernel(const int32_t* __restrict__ tok_src,
                                                              const uint4* __restrict__ hid_src,
                                                              int32_t* __restrict__ tok_dst,
                                                              uint4* __restrict__ hid_dst, int B, int n16) {
  pdl_wait_prior_grid();
  pdl_launch_dependents();  // the input stage may start its weight stream now
  const int base = blockIdx.x * kIoThreads * kIoPer + threadIdx.x;
  uint4 v[kIoPer];
#pragma unroll
  for (int j = 0; j < kIoPer; ++j)
    if (base + j * kIoThreads < n16) v[j] = hid_src[base + j * kIoThreads];
#pragma unroll
  for (int j = 0; j < kIoPer; ++j)
    if (base + j * kIoThreads < n16) hid_dst[base + j * kIoThreads] = v[j];
  if (blockIdx.x == 0 && threadIdx.x < B) tok_dst[threadIdx.x] = tok_src[threadIdx.x];
}

// One thread writes the drafts and the status into host memory, makes them visible to the host
// (system-scope fence), then copies the call's sequence number (seq_in, set by the host before
// the launch) to seq_out, which the host polls instead of waiting for the stream (may be null).
__global__ void __launch_bounds__(32) host_out_kernel(const int32_t* draft_src, int32_t* draft_dst,
                                                      const int32_t* status_src, int32_t* status_dst, int B,
                                                      const uint32_t* seq_in, uint32_t* seq_out) {
  pdl_wait_prior_grid();  // the draft comes from the sweep
  if (threadIdx.x == 0) {
    for (int b = 0; b < B; ++b) draft_dst[b] = draft_src[b];
    if (status_src != nullptr) *status_dst = *status_src;
    __threadfence_system();
    if (seq_out != nullptr) *reinterpret_cast<volatile uint32_t*>(seq_out) = *reinterpret_cast<const volatile uint32_t*>(seq_in);
  }
}

}  // namespace

cudaError_t launch_host_in(const int32_t* tok_src, const uint16_t* hid_src, int32_t* tok_dst, uint16_t* hid_dst,
                           int B, int H, cudaStream_t stream) {
  DeviceInfo di;
  cudaError_t err = device_info(&di);
  if (err != cudaSuccess) return err;
  int n16 = static_cast<int>(static_cast<int64_t>(B) * H * 2 / 16);
  const void* src = hid_src;
  void* dst = hid_dst;
  void* params[] = {&tok_src, &src, &tok_dst, &dst, &B, &n16};
  const int grid = (n16 + kIoThreads * kIoPer - 1) / (kIoThreads * kIoPer);
  return launch_pdl(reinterpret_cast<const void*>(host_in_kernel), dim3(grid > 0 ? grid : 1), dim3(kIoThreads), 0,
                    stream, params);
}

cudaError_t launch_host_out(const int32_t* draft_src, int32_t* draft_dst, const int32_t* status_src, int32_t* status_dst,
                            int B, const uint32_t* seq_in, uint32_t* seq_out, cudaStream_t stream) {
  DeviceInfo di;
  cudaError_t err = device_info(&di);
  if (err != cudaSuccess) return err;
  void* params[] = {&draft_src, &draft_dst, &status_src, &status_dst, &B, &seq_in, &seq_out};
  return launch_pdl(reinterpret_cast<const void*>(host_out_kernel), dim3(1), dim3(32), 0, stream, params);
}

}  // namespace mtp
