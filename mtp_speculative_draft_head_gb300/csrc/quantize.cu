// FP8 E4M3 copy of the lm_head ("glm5next_mtp_head.rs", `head_fp8` doc: an E4M3 copy of the
// head used for drafting only; the pages do not print the scale scheme, so the build uses one
// FP32 scale per row):
//   s[v]    = fp32( max_k |w[v, k]| / 448 )
//   q[v, k] = e4m3_rne_satfinite( fp32( w[v, k] / s[v] ) )     (s = 0: all codes 0)
// Both divisions are IEEE round-to-nearest (no fast-math in this file), and the E4M3 rounding
// is the hardware conversion with satfinite, so the codes are a pure function of the input.
// Run once per weight load, not per draft: one warp per row, two passes over the row.
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

namespace mtp {

namespace {

__device__ __forceinline__ uint8_t e4m3_of(float q) {
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(q, __NV_SATFINITE, __NV_E4M3));
}

__global__ void __launch_bounds__(256) quantize_kernel(const uint16_t* __restrict__ w,
                                                       uint8_t* __restrict__ q,
                                                       float* __restrict__ scale,
                                                       int32_t* __restrict__ status, int64_t V,
                                                       int H) {
  const int lane = threadIdx.x & 31;
  const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t tw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const bool vec = (H & 15) == 0;
  for (int64_t v = gw; v < V; v += tw) {
    const uint16_t* row = w + v * H;
    uint8_t* qrow = q + v * H;
    // pass 1: magnitude maximum on the bit patterns (|x| order == (bits & 0x7FFF) order for
    // finite BF16) and a non-finite flag
    uint32_t mx = 0, bad = 0;
    if (vec) {
      const uint4* rv = reinterpret_cast<const uint4*>(row);
      for (int j = lane; j < H / 8; j += 32) {
        const uint4 u = rv[j];
        const uint32_t ws[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const uint32_t lo = ws[t] & 0x7FFFu, hi = (ws[t] >> 16) & 0x7FFFu;
          bad |= ((lo & 0x7F80u) == 0x7F80u) | ((hi & 0x7F80u) == 0x7F80u);
          mx = max(mx, max(lo, hi));
        }
      }
    } else {
      for (int k = lane; k < H; k += 32) {
        const uint32_t m = row[k] & 0x7FFFu;
        bad |= (m & 0x7F80u) == 0x7F80u;
        mx = max(mx, m);
      }
    }
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) {
      mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, m));
      bad |= __shfl_xor_sync(0xffffffffu, bad, m);
    }
    float s = __fdiv_rn(bf16_bits_to_f32(mx), 448.0f);
    if (bad) {
      if (lane == 0) store_status(status, MTP_ERR_NONFINITE);
      s = 0.0f;
    }
    if (lane == 0) scale[v] = s;
    // pass 2: codes
    if (vec) {
      const uint4* rv = reinterpret_cast<const uint4*>(row);
      uint4* qv = reinterpret_cast<uint4*>(qrow);
      for (int j = lane; j < H / 16; j += 32) {
        const uint4 u0 = rv[2 * j], u1 = rv[2 * j + 1];
        const uint32_t ws[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
        uint32_t out[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          uint32_t word = 0;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t pair = ws[2 * t + h];
            const uint32_t c0 = (s == 0.0f) ? 0u : e4m3_of(__fdiv_rn(bf16_lo(pair), s));
            const uint32_t c1 = (s == 0.0f) ? 0u : e4m3_of(__fdiv_rn(bf16_hi(pair), s));
            word |= (c0 | (c1 << 8)) << (16 * h);
          }
          out[t] = word;
        }
        qv[j] = make_uint4(out[0], out[1], out[2], out[3]);
      }
    } else {
      for (int k = lane; k < H; k += 32)
        qrow[k] = (s == 0.0f) ? uint8_t(0) : e4m3_of(__fdiv_rn(bf16_bits_to_f32(row[k]), s));
    }
  }
}

}  // namespace

cudaError_t launch_quantize(const uint16_t* w, uint8_t* q, float* scale, int32_t* status, int V,
                            int H, cudaStream_t stream) {
  DeviceInfo di;
  cudaError_t err = device_info(&di);
  if (err != cudaSuccess) return err;
  const int64_t warps_wanted = V;
  int64_t blocks = (warps_wanted + 7) / 8;
  const int64_t cap = static_cast<int64_t>(di.sm_count) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, quantize_kernel, w, q, scale, status, static_cast<int64_t>(V), H);
}

}  // namespace mtp
