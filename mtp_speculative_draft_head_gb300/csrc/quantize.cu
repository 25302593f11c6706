// FP8 E4M3 copy of the lm_head ("glm5next_mtp_head.rs", `head_fp8` doc: an E4M3 copy of the
// head used for drafting only; the pages do not print the scale scheme, so the build uses one
// FP32 scale per row):
//   s[v]    = fp32( max_k |w[v, k]| / 448 )
//   q[v, k] = e4m3_rne_satfinite( fp32( w[v, k] / s[v] ) )     (s = 0: all codes 0)
// Both divisions are IEEE round-to-nearest (no fast-math in this file), and the E4M3 rounding
// is the hardware conversion with satfinite, so the codes are a pure function of the input.
// Run once per weight load, not per draft: one warp per row, two passes over the row (the
// second from L2), with several 16-byte loads in flight per lane in the first.
//
// The codes without a division per element. The code of the quotient depends only on which
// pair of neighbouring E4M3 rounding boundaries the quotient lies between. With r = 1/s, the
// products y_up = f * r (1 + 2^-21) and y_dn = f * r (1 - 2^-21) (each factor and product
// rounded to nearest) bracket fp32(f / s) strictly: the four roundings move them by at most
// 3 * 2^-24 relative, fp32(f / s) is within 2^-24 of f / s, and 2^-21 - 3 * 2^-24 > 2^-24.
// The conversion to E4M3 (round to nearest even, saturating) is monotonic, so when y_up and
// y_dn give the same code, fp32(f / s) gives it too. Otherwise (a boundary inside the bracket:
// nearly always an exact tie, about 0.5 % of the elements of Gaussian rows) the code comes from
// the division itself. Quotients below the
// fp32 normal range convert to a signed zero on all three paths. Rows whose scale is not a
// normal fp32 number take the division for every element.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

namespace mtp {

namespace {

constexpr int kQThreads = 256;
// Measured at H = 6144, V = 154880 (best of 7 runs): 4 loads, 1 piece, 6 blocks per SM (40
// registers, 48 warps per SM) 517 us; 8 / 2 / 4 blocks 524 us; 8 / 4 / no minimum (75 registers)
// 598 us; 16 / 8 / no minimum 1687 us. More warps beat more loads in flight per warp.
#ifndef MTP_Q_LOADS
#define MTP_Q_LOADS 4
#endif
#ifndef MTP_Q_PIECES
#define MTP_Q_PIECES 1
#endif
#ifndef MTP_Q_MINB
#define MTP_Q_MINB 6
#endif
constexpr int kLoadsMag = MTP_Q_LOADS;     // 16-byte loads in flight per lane, magnitude pass
constexpr int kPiecesCode = MTP_Q_PIECES;  // 16-element pieces (32 bytes in, 16 out) per lane and step

// Two E4M3 codes (round to nearest even, satfinite): byte 0 from lo, byte 1 from hi.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}

// max of the two 16-bit halves, lane by lane
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Codes of one bf16 pair (32-bit word) through the bracket, the division when it is open.
__device__ __forceinline__ uint32_t pair_codes(uint32_t pair, float s, float r_up, float r_dn) {
  const float a = bf16_lo(pair), b = bf16_hi(pair);
  const uint32_t up = e4m3x2(__fmul_rn(a, r_up), __fmul_rn(b, r_up));
  const uint32_t dn = e4m3x2(__fmul_rn(a, r_dn), __fmul_rn(b, r_dn));
  if (up == dn) return up;
  return e4m3x2(__fdiv_rn(a, s), __fdiv_rn(b, s));
}

__device__ __forceinline__ uint32_t pair_codes_div(uint32_t pair, float s) {
  return e4m3x2(__fdiv_rn(bf16_lo(pair), s), __fdiv_rn(bf16_hi(pair), s));
}

// Rows with H % 16 == 0: 16-byte loads and stores.
__global__ void __launch_bounds__(kQThreads, MTP_Q_MINB) quantize_vec_kernel(const uint16_t* __restrict__ w,
                                                                 uint8_t* __restrict__ q,
                                                                 float* __restrict__ scale,
                                                                 int32_t* __restrict__ status,
                                                                 int64_t V, int H) {
  const int lane = threadIdx.x & 31;
  const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t tw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int n8 = H >> 3;    // 16-byte words of a row
  const int n16 = H >> 4;   // 16-element pieces of a row
  for (int64_t v = gw; v < V; v += tw) {
    const uint4* rv = reinterpret_cast<const uint4*>(w + v * H);
    // pass 1: magnitude maximum on the bit patterns (|x| order == (bits & 0x7FFF) order for
    // finite BF16; NaN and Inf have the largest patterns, so they show in the maximum)
    uint32_t mx2 = 0;
    for (int b = 0; b < n8; b += 32 * kLoadsMag) {
      uint4 u[kLoadsMag];
#pragma unroll
      for (int i = 0; i < kLoadsMag; ++i) {
        const int j = b + 32 * i + lane;
        u[i] = j < n8 ? rv[j] : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int i = 0; i < kLoadsMag; ++i) {
        mx2 = max_u16x2(mx2, u[i].x & 0x7FFF7FFFu);
        mx2 = max_u16x2(mx2, u[i].y & 0x7FFF7FFFu);
        mx2 = max_u16x2(mx2, u[i].z & 0x7FFF7FFFu);
        mx2 = max_u16x2(mx2, u[i].w & 0x7FFF7FFFu);
      }
    }
    uint32_t mx = max(mx2 & 0xFFFFu, mx2 >> 16);
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, m));
    float s = __fdiv_rn(bf16_bits_to_f32(mx), 448.0f);
    if (mx >= 0x7F80u) {  // a NaN or Inf in the row
      if (lane == 0) store_status(status, MTP_ERR_NONFINITE);
      s = 0.0f;
    }
    if (lane == 0) scale[v] = s;
    // pass 2: codes
    uint4* qv = reinterpret_cast<uint4*>(q + v * H);
    const bool bracket = s >= 1.17549435e-38f;  // a normal scale: 1/s is finite and exact to 2^-24
    const float r = bracket ? __frcp_rn(s) : 0.0f;
    const float r_up = __fmul_rn(r, 1.0f + 0x1p-21f), r_dn = __fmul_rn(r, 1.0f - 0x1p-21f);
    for (int b = 0; b < n16; b += 32 * kPiecesCode) {
      uint4 u0[kPiecesCode], u1[kPiecesCode];
#pragma unroll
      for (int i = 0; i < kPiecesCode; ++i) {
        const int j = b + 32 * i + lane;
        if (j < n16) {
          u0[i] = __ldcs(rv + 2 * j);
          u1[i] = __ldcs(rv + 2 * j + 1);
        }
      }
#pragma unroll
      for (int i = 0; i < kPiecesCode; ++i) {
        const int j = b + 32 * i + lane;
        if (j >= n16) continue;
        const uint32_t ws[8] = {u0[i].x, u0[i].y, u0[i].z, u0[i].w, u1[i].x, u1[i].y, u1[i].z, u1[i].w};
        uint32_t c[8];
        if (s == 0.0f) {
#pragma unroll
          for (int t = 0; t < 8; ++t) c[t] = 0u;
        } else if (bracket) {
#pragma unroll
          for (int t = 0; t < 8; ++t) c[t] = pair_codes(ws[t], s, r_up, r_dn);
        } else {
#pragma unroll
          for (int t = 0; t < 8; ++t) c[t] = pair_codes_div(ws[t], s);
        }
        __stcs(qv + j, make_uint4(c[0] | (c[1] << 16), c[2] | (c[3] << 16), c[4] | (c[5] << 16),
                                  c[6] | (c[7] << 16)));
      }
    }
  }
}

// Any H: one element at a time.
__global__ void __launch_bounds__(kQThreads) quantize_scalar_kernel(const uint16_t* __restrict__ w,
                                                                    uint8_t* __restrict__ q,
                                                                    float* __restrict__ scale,
                                                                    int32_t* __restrict__ status,
                                                                    int64_t V, int H) {
  const int lane = threadIdx.x & 31;
  const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t tw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t v = gw; v < V; v += tw) {
    const uint16_t* row = w + v * H;
    uint8_t* qrow = q + v * H;
    uint32_t mx = 0;
    for (int k = lane; k < H; k += 32) mx = max(mx, static_cast<uint32_t>(row[k]) & 0x7FFFu);
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, m));
    float s = __fdiv_rn(bf16_bits_to_f32(mx), 448.0f);
    if (mx >= 0x7F80u) {
      if (lane == 0) store_status(status, MTP_ERR_NONFINITE);
      s = 0.0f;
    }
    if (lane == 0) scale[v] = s;
    for (int k = lane; k < H; k += 32)
      qrow[k] = (s == 0.0f) ? uint8_t(0)
                            : static_cast<uint8_t>(e4m3x2(__fdiv_rn(bf16_bits_to_f32(row[k]), s), 0.0f));
  }
}

}  // namespace

cudaError_t launch_quantize(const uint16_t* w, uint8_t* q, float* scale, int32_t* status, int V,
                            int H, cudaStream_t stream) {
  DeviceInfo di;
  cudaError_t err = device_info(&di);
  if (err != cudaSuccess) return err;
  const bool vec = (H & 15) == 0;
  const void* kern = vec ? reinterpret_cast<const void*>(quantize_vec_kernel)
                         : reinterpret_cast<const void*>(quantize_scalar_kernel);
  int per_sm = 0;
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kQThreads, 0);
  if (err != cudaSuccess) return err;
  const int64_t warps_wanted = V;
  int64_t blocks = (warps_wanted + kQThreads / 32 - 1) / (kQThreads / 32);
  const int64_t cap = static_cast<int64_t>(di.sm_count) * (per_sm > 0 ? per_sm : 1);
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  int64_t V64 = V;
  void* args[] = {&w, &q, &scale, &status, &V64, &H};
  return cudaLaunchKernel(kern, dim3(static_cast<unsigned>(blocks)), dim3(kQThreads), args, 0, stream);
}

}  // namespace mtp
