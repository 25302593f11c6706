// Device building blocks shared by the MTP-head kernels (sm_103a).
//
//  * PTX wrappers: mbarrier, 1-D bulk async copy (TMA engine, global -> shared), L2 eviction
//    policy, async-proxy fence, programmatic dependent launch, global timer.
//  * Exact-rounding numerics: TwoSum, double-float accumulation, BF16 round-to-nearest-even
//    of a double-float value, the E4M3 bit-placement decode.
//  * Packed f32x2 arithmetic and packed double-float accumulation.
//  * The RMSNorm prologue (rms_norm_vanilla, x * w / rms) for several vectors, into shared memory.
//  * The (max, lowest index) argmax combine.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mtp_head.h"

namespace mtp {

constexpr int kMaxB = 16;        // sequences per sweep
constexpr int kMaxGrid = 1024;   // CTAs per launch (bounds the workspace)
constexpr int kWsHeader = 128;   // workspace bytes before the per-CTA partials
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // give up a wait after 2 s

// ------------------------------------------------------------------------------------------
// PTX wrappers
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Wait for phase `parity` of an mbarrier, giving up after kWaitLimitNs. Returns false on
// timeout; the caller records MTP_ERR_TIMEOUT and stops.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
  return true;
}

// L2 policy for data read exactly once per pass (weights far larger than L2).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// 1-D bulk copy global -> shared through the TMA engine, completing `bytes` transaction bytes
// on mbarrier `bar`. Requires 16-byte aligned addresses and a size that is a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// Programmatic dependent launch: wait for the preceding grid (no-op when the launch did not
// ask for it), and allow the next grid to be scheduled.
__device__ __forceinline__ void pdl_wait_prior_grid() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void store_status(int32_t* status, int32_t code) {
  if (status != nullptr) atomicCAS(reinterpret_cast<int*>(status), 0, code);
}

// ------------------------------------------------------------------------------------------
// Numerics
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b16) { return __uint_as_float(b16 << 16); }
__device__ __forceinline__ float bf16_lo(uint32_t pair) { return __uint_as_float(pair << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t pair) { return __uint_as_float(pair & 0xFFFF0000u); }

// s + e == a + b exactly (Knuth's TwoSum; no ordering requirement on |a|, |b|).
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bp = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bp)), __fsub_rn(b, bp));
}

// Double-float value hi + lo.
struct DF {
  float hi, lo;
};

__device__ __forceinline__ void df_add(DF& acc, float g) {
  float s, e;
  two_sum(acc.hi, g, s, e);
  acc.hi = s;
  acc.lo = __fadd_rn(acc.lo, e);
}

__device__ __forceinline__ DF df_add(DF a, DF b) {
  float s, e;
  two_sum(a.hi, b.hi, s, e);
  e = __fadd_rn(e, __fadd_rn(a.lo, b.lo));
  DF r;
  two_sum(s, e, r.hi, r.lo);
  return r;
}

__device__ __forceinline__ DF shfl_xor_df(DF v, int m) {
  DF r;
  r.hi = __shfl_xor_sync(0xffffffffu, v.hi, m);
  r.lo = __shfl_xor_sync(0xffffffffu, v.lo, m);
  return r;
}

// Round the exact value hi + lo to the nearest BF16 (ties to even). After renormalising,
// hi holds the value rounded to fp32 and lo the exact remainder (|lo| <= half an fp32 ulp), so
// only a hi that sits exactly on a BF16 midpoint needs lo to decide.
__device__ __forceinline__ uint16_t bf16_rne_df(float hi, float lo) {
  float s, e;
  two_sum(hi, lo, s, e);
  const uint32_t u = __float_as_uint(s);
  if ((u & 0x7F800000u) == 0x7F800000u) {  // inf or NaN
    if (u & 0x007FFFFFu) return static_cast<uint16_t>(((u >> 16) & 0x8000u) | 0x7FC0u);
    return static_cast<uint16_t>(u >> 16);
  }
  const uint32_t rem = u & 0xFFFFu;
  const uint32_t base = u >> 16;
  bool up;
  if (rem > 0x8000u) {
    up = true;
  } else if (rem < 0x8000u) {
    up = false;
  } else if (e == 0.0f) {
    up = (base & 1u) != 0u;
  } else {
    up = ((__float_as_uint(e) ^ u) & 0x80000000u) == 0u;  // same sign: larger magnitude
  }
  return static_cast<uint16_t>(base + (up ? 1u : 0u));
}

// E4M3 byte i (0..3) of a 32-bit word -> fp32 holding value * 2^-120, exactly.
// The byte S.EEEE.MMM is placed as fp32 sign S, exponent field 0000EEEE and mantissa MMM:
// exponent field E gives 2^(E-127) * 1.MMM = 2^-120 * 2^(E-7) * 1.MMM; field 0 gives the fp32
// subnormal 2^-126 * MMM/8 = 2^-120 * 2^-6 * MMM/8 -- the E4M3 subnormal scaled the same way.
// (The NaN code S.1111.111 is never produced by the quantiser and decodes to a finite value.)
template <int I>
__device__ __forceinline__ float e4m3_byte_scaled(uint32_t w) {
  const int32_t t = static_cast<int32_t>(w << (24 - 8 * I)) >> 4;  // arithmetic shift
  return __uint_as_float(static_cast<uint32_t>(t) & 0x87F00000u);
}
constexpr float kE4m3Unscale = 1.329227995784915872903807060280344576e36f;  // 2^120

// ------------------------------------------------------------------------------------------
// Argmax: (value, index) pairs; larger value wins, equal values -> lower index, NaN never wins,
// index -1 marks "nothing yet".
// ------------------------------------------------------------------------------------------
struct ArgBest {
  float v;
  int32_t i;
};

__device__ __forceinline__ bool arg_beats(float v, int32_t i, const ArgBest& b) {
  if (v != v) return false;
  if (b.i < 0) return i >= 0;
  return v > b.v || (v == b.v && i < b.i);
}

__device__ __forceinline__ void arg_update(ArgBest& b, float v, int32_t i) {
  if (arg_beats(v, i, b)) {
    b.v = v;
    b.i = i;
  }
}

// ------------------------------------------------------------------------------------------
// Packed fp32 pairs (sm_100+ f32x2 instructions): two IEEE round-to-nearest operations per
// instruction, lane-wise identical to the scalar ones.
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float f2_lo(uint64_t v) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
  return lo;
}
__device__ __forceinline__ float f2_hi(uint64_t v) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
  return hi;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// BF16 pair (low half first) -> {f32(low), f32(high)}
__device__ __forceinline__ uint64_t bf16x2_to_f2(uint32_t u) {
  return f2_pack(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
}

// Two independent double-floats, packed: (hi.x, lo.x) and (hi.y, lo.y).
struct DF2 {
  uint64_t hi, lo;
};
// TwoSum of each lane's (hi, p), the error added to lo.
__device__ __forceinline__ void df2_add(DF2& a, uint64_t p) {
  const uint64_t s = f2_add(a.hi, p);
  const uint64_t bp = f2_sub(s, a.hi);
  const uint64_t e = f2_add(f2_sub(a.hi, f2_sub(s, bp)), f2_sub(p, bp));
  a.hi = s;
  a.lo = f2_add(a.lo, e);
}
__device__ __forceinline__ DF df2_x(const DF2& a) { return DF{f2_lo(a.hi), f2_lo(a.lo)}; }
__device__ __forceinline__ DF df2_y(const DF2& a) { return DF{f2_hi(a.hi), f2_hi(a.lo)}; }

// ------------------------------------------------------------------------------------------
// rms_norm_vanilla prologue for several vectors at once:
//   out_j = bf16( x_j * w_j / sqrt(mean(x_j^2) + eps) ), written into shared memory at layout(k).
// The sums of squares are double-floats (each square of a BF16 value is exact in fp32), 1/rms is
// formed in fp64 and split into two fp32 parts, and x*w (exact in fp32) times 1/rms is rounded
// once to BF16 from a double-float -- so each output is the correctly rounded BF16 of the fp64
// expression unless that lies within ~2^-40 relative of a rounding midpoint.
// One pass over the inputs, one block reduction for all vectors. All NT threads of the block
// call it; `red` holds >= njobs * (2 * NT / 32 + 2) floats. A job with valid == false writes
// zeros without reading x.
// ------------------------------------------------------------------------------------------
struct NormJob {
  const uint16_t* x;
  const uint16_t* w;
  uint16_t* out;
  bool valid;
};

template <int NT, class Layout, class JobFn>
__device__ void rms_norm_multi_to_smem(int njobs, int n, float eps, float* red, JobFn job,
                                       Layout layout) {
  constexpr int NW = NT / 32;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int j = 0; j < njobs; ++j) {
    const NormJob J = job(j);
    DF acc{0.0f, 0.0f};
    if (J.valid) {
      const bool vec = ((n & 7) == 0) && ((reinterpret_cast<uintptr_t>(J.x) & 15u) == 0);
      if (vec) {
        const uint4* xv = reinterpret_cast<const uint4*>(J.x);
        for (int v = tid; v < n / 8; v += NT) {
          const uint4 q = xv[v];
          const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const float a = bf16_lo(u[t]), b = bf16_hi(u[t]);
            df_add(acc, __fmul_rn(a, a));
            df_add(acc, __fmul_rn(b, b));
          }
        }
      } else {
        for (int k = tid; k < n; k += NT) {
          const float a = bf16_bits_to_f32(J.x[k]);
          df_add(acc, __fmul_rn(a, a));
        }
      }
    }
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) acc = df_add(acc, shfl_xor_df(acc, m));
    if (lane == 0) {
      red[(j * NW + warp) * 2] = acc.hi;
      red[(j * NW + warp) * 2 + 1] = acc.lo;
    }
  }
  __syncthreads();
  float* rr = red + njobs * NW * 2;
  for (int j = tid; j < njobs; j += NT) {
    DF tot{red[j * NW * 2], red[j * NW * 2 + 1]};
    for (int i = 1; i < NW; ++i) tot = df_add(tot, DF{red[(j * NW + i) * 2], red[(j * NW + i) * 2 + 1]});
    const double ms = (static_cast<double>(tot.hi) + static_cast<double>(tot.lo)) / static_cast<double>(n);
    const double r = 1.0 / sqrt(ms + static_cast<double>(eps));
    const float rh = static_cast<float>(r);
    rr[2 * j] = rh;
    rr[2 * j + 1] = static_cast<float>(r - static_cast<double>(rh));
  }
  __syncthreads();
  for (int j = 0; j < njobs; ++j) {
    const NormJob J = job(j);
    const float rh = rr[2 * j], rl = rr[2 * j + 1];
    const bool vec = ((n & 7) == 0) && ((reinterpret_cast<uintptr_t>(J.x) & 15u) == 0) &&
                     ((reinterpret_cast<uintptr_t>(J.w) & 15u) == 0);
    if (vec) {
      for (int v = tid; v < n / 8; v += NT) {
        uint32_t o[4] = {0u, 0u, 0u, 0u};
        if (J.valid) {
          const uint4 xq = reinterpret_cast<const uint4*>(J.x)[v];
          const uint4 wq = reinterpret_cast<const uint4*>(J.w)[v];
          const uint32_t xu[4] = {xq.x, xq.y, xq.z, xq.w}, wu[4] = {wq.x, wq.y, wq.z, wq.w};
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            uint32_t half[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const float xe = h ? bf16_hi(xu[t]) : bf16_lo(xu[t]);
              const float we = h ? bf16_hi(wu[t]) : bf16_lo(wu[t]);
              const float p = __fmul_rn(xe, we);  // exact
              const float yh = __fmul_rn(p, rh);
              const float yl = __fmaf_rn(p, rl, __fmaf_rn(p, rh, -yh));
              half[h] = bf16_rne_df(yh, yl);
            }
            o[t] = half[0] | (half[1] << 16);
          }
        }
        // 8 consecutive elements starting at a multiple of 8 stay consecutive in every layout
        *reinterpret_cast<uint4*>(J.out + layout(8 * v)) = make_uint4(o[0], o[1], o[2], o[3]);
      }
    } else {
      for (int k = tid; k < n; k += NT) {
        uint16_t o = 0;
        if (J.valid) {
          const float p = __fmul_rn(bf16_bits_to_f32(J.x[k]), bf16_bits_to_f32(J.w[k]));
          const float yh = __fmul_rn(p, rh);
          const float yl = __fmaf_rn(p, rl, __fmaf_rn(p, rh, -yh));
          o = bf16_rne_df(yh, yl);
        }
        J.out[layout(k)] = o;
      }
    }
  }
}

// Shared-memory index of element k of a vector when weight vectors hold 16 elements (FP8) and
// a lane reads the matching 32 bytes of BF16 activations as two 16-byte slots: slots of 32
// consecutive weight vectors are interleaved so both reads of a warp are conflict-free.
struct LayoutIdentity {
  __device__ __forceinline__ int operator()(int k) const { return k; }
};
struct LayoutFp8 {
  __device__ __forceinline__ int operator()(int k) const {
    const int J = k >> 4, e = k & 15;
    const int slot = (J >> 5) * 64 + ((e >> 3) << 5) + (J & 31);
    return slot * 8 + (e & 7);
  }
};

}  // namespace mtp
