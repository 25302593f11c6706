// Pick over vocabulary shards ("glm5next_mtp_head.rs", `forward_one`, sharded branch: every rank
// sweeps its own row range of lm_head, then the ranks' (max logit, index) pairs decide the draft,
// the lower range winning a tie). Each shard's output stage stored one exchange key per sequence
// (pick.h: the argmax order as the signed order of int64), so the pick is the maximum of the
// keys: R keys per sequence, one warp per sequence, a shuffle tree, one decode.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

namespace mtp {

namespace {

__global__ void __launch_bounds__(kMaxB * 32) pick_combine_kernel(const int64_t* picks, int R, int B,
                                                                   int32_t* draft, float* value) {
  pdl_wait_prior_grid();  // the keys come from the preceding kernels
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int b = warp; b < B; b += blockDim.x >> 5) {
    long long k = kPickEmpty;
    for (int r = lane; r < R; r += 32) {
      const long long o = __ldcg(reinterpret_cast<const long long*>(picks) + static_cast<size_t>(r) * B + b);
      k = o > k ? o : k;
    }
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) {
      const long long o = __shfl_xor_sync(0xffffffffu, k, m);
      k = o > k ? o : k;
    }
    if (lane == 0) {
      draft[b] = pick_index(k);
      if (value != nullptr) value[b] = pick_value(k);
    }
  }
  pdl_launch_dependents();
}

}  // namespace

cudaError_t launch_pick_combine(const int64_t* picks, int R, int B, int32_t* draft, float* value,
                                cudaStream_t stream) {
  DeviceInfo di;
  cudaError_t err = device_info(&di);
  if (err != cudaSuccess) return err;
  const int warps = B < kMaxB ? B : kMaxB;
  void* args[] = {&picks, &R, &B, &draft, &value};
  return launch_pdl(reinterpret_cast<const void*>(pick_combine_kernel), dim3(1), dim3(warps * 32), 0, stream,
                    args);
}

}  // namespace mtp
