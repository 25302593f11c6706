// Output stage of the MTP draft head: shared_head.norm, the lm_head vocabulary sweep and the
// argmax, fused into one kernel ("glm5next_mtp_head.rs", `forward_one`: `norm` of x with
// final_norm in place, `dense_gemv` / `dense_gemv_fp8w` over the vocabulary, `argmax_bf16`).
//
// Design (one GB300, HBM-bound GEMV, no tensor cores at these batch sizes):
//  * Persistent grid: one CTA per SM, each owning a contiguous range of vocabulary rows (V split
//    evenly, so the tail is at most one row per CTA).
//  * Each warp streams its own rows through a private ring of shared-memory stages filled by
//    1-D bulk async copies (TMA engine, `cp.async.bulk` + mbarrier transaction counts, L2
//    evict-first). The weight stream never passes through registers on its way to shared
//    memory, so eight warps keep ~200 KB per SM in flight.
//  * Before waiting for the preceding kernel (programmatic dependent launch) each warp already
//    issues its first stages: the weights do not depend on x.
//  * Prologue: every CTA computes xhat = rms_norm_vanilla(x, final_norm_w) for its B sequences
//    into shared memory (BF16). For one sequence at the GLM sizes a lane then keeps the part of
//    xhat it multiplies in registers, a stage holds a whole row and rows are reduced eight at a
//    time; otherwise xhat stays in shared memory (laid out so the per-lane reads are bank-
//    conflict free) and rows are staged in 4 KB chunks.
//  * Each row is reduced by one warp with a fixed lane->element map and a fixed lane tree, so
//    identical rows give bit-identical logits (exact ties stay exact).
//  * FP8 E4M3 codes are widened exactly: by the hardware E4M3 -> f16 conversion (activations then
//    held as f16 scaled by a power of two), or by bit placement into a BF16 word holding the
//    value times 2^-120. Either way products are exact and the row sum is scaled back by a power
//    of two (exact) and by the row scale.
//  * Epilogue: FP32 logits written once (optional), a per-warp then per-CTA (max, lowest index)
//    and a last-CTA-done combine of the per-CTA partials into draft[b]. No CTA ever waits for
//    another; the counter returns itself to zero for the next call or graph replay.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "host_back.h"

namespace mtp {

namespace {

// ------------------------------------------------------------------------------------------
// Per-CTA epilogue: combine warp bests, publish the CTA partial, and let the last CTA finish.
// best[] is uniform across the lanes of a warp.
// ------------------------------------------------------------------------------------------
// hb (a recorded host-buffer step, else null): the last CTA also hands the drafts and the status
// back to mapped host memory, then sets the completion word the host polls.
template <int NB>
__device__ void argmax_finish(const ArgBest* best, int nb, ArgBest* wbest, const SweepArgs& a,
                              const HostBack* hb = nullptr) {
  uint8_t* ws = a.ws;
  __shared__ int is_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  if (lane == 0) {
#pragma unroll
    for (int b = 0; b < NB; ++b)
      if (b < nb) wbest[warp * nb + b] = best[b];
  }
  __syncthreads();
  unsigned int* counter = reinterpret_cast<unsigned int*>(ws);
  if (threadIdx.x < nb) {
    ArgBest c{0.0f, -1};
    for (int w = 0; w < nwarps; ++w) {
      const ArgBest o = wbest[w * nb + threadIdx.x];
      if (o.i >= 0) arg_update(c, o.v, o.i);
    }
    pick_publish(ws, threadIdx.x, c.v, c.i, a.index_base);
    __threadfence();
  }
  __syncthreads();
  if (threadIdx.x == 0) is_last = (atomicAdd(counter, 1u) == gridDim.x - 1) ? 1 : 0;
  __syncthreads();
  if (is_last) {
    __threadfence();
    if (threadIdx.x < nb) pick_finish(ws, threadIdx.x, a.draft, a.pick);
    if (hb != nullptr) {
      if (static_cast<int>(threadIdx.x) < nb) {
        hb->draft[threadIdx.x] = a.draft[threadIdx.x];  // written by this thread just above
        __threadfence_system();
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        volatile uint32_t* w = hb->words;
        if (a.status != nullptr) w[0] = static_cast<uint32_t>(*reinterpret_cast<const volatile int32_t*>(a.status));
        __threadfence_system();
        w[3] = w[2];
      }
    }
    if (threadIdx.x == 0) {
      // every CTA has finished claiming rows: ready for the next launch
      atomicExch(reinterpret_cast<unsigned int*>(ws + kRowCounterOffset), 0u);
      atomicExch(counter, 0u);
    }
  }
}

// Mixed-precision FMA: acc0 += lo(w) * lo(x), acc1 += hi(w) * hi(x) for BF16 pairs, each with
// the exact product and one fp32 rounding (the same value as an fp32 FMA of the widened halves).
__device__ __forceinline__ void fma2_bf16(float& acc0, float& acc1, uint32_t w, uint32_t x) {
  asm("{\n\t.reg .b16 wl, wh, xl, xh;\n\t"
      "mov.b32 {wl, wh}, %2;\n\t"
      "mov.b32 {xl, xh}, %3;\n\t"
      "fma.rn.f32.bf16 %0, wl, xl, %0;\n\t"
      "fma.rn.f32.bf16 %1, wh, xh, %1;\n\t}"
      : "+f"(acc0), "+f"(acc1)
      : "r"(w), "r"(x));
}

// BF16 pair FMA into two accumulators, either with the mixed-precision instruction or by
// widening both pairs to fp32 (identical results).
template <bool kMixed>
__device__ __forceinline__ void fma_pair(float& acc0, float& acc1, uint32_t w, uint32_t x) {
  if constexpr (kMixed) {
    fma2_bf16(acc0, acc1, w, x);
  } else {
    acc0 = __fmaf_rn(bf16_lo(w), bf16_lo(x), acc0);
    acc1 = __fmaf_rn(bf16_hi(w), bf16_hi(x), acc1);
  }
}

// Four E4M3 codes -> two BF16 pairs holding value * 2^-120 (sign to bit 15, magnitude bits
// EEEE.MMM to bits 10..4 of each half: BF16 exponent field 0000EEEE, mantissa MMM0000).
// Per half: the code c = S.mag placed at bits 15..8 reads S<<15 | mag<<8; subtracting 240*mag
// leaves S<<15 | mag<<4 (never negative, so no borrow crosses into the other half).
__device__ __forceinline__ void e4m3x4_to_bf16x2x2(uint32_t w, uint32_t& p01, uint32_t& p23) {
  const uint32_t m = w & 0x7F7F7F7Fu;
  p01 = __byte_perm(w, 0u, 0x1404u) - 240u * __byte_perm(m, 0u, 0x4140u);
  p23 = __byte_perm(w, 0u, 0x3424u) - 240u * __byte_perm(m, 0u, 0x4342u);
}

// One 16-byte vector of 16 E4M3 codes times the 16 matching BF16 activations (8 pairs x[0..7]),
// elements 2i -> acc0, 2i+1 -> acc1 (bit-placement decode, values * 2^-120).
template <bool kMixed>
__device__ __forceinline__ void fp8_dot16(const uint4& q, const uint32_t* x, float& acc0, float& acc1) {
  const uint32_t qu[4] = {q.x, q.y, q.z, q.w};
  if constexpr (kMixed) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      uint32_t p01, p23;
      e4m3x4_to_bf16x2x2(qu[u], p01, p23);
      fma2_bf16(acc0, acc1, p01, x[2 * u]);
      fma2_bf16(acc0, acc1, p23, x[2 * u + 1]);
    }
  } else {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      acc0 = __fmaf_rn(e4m3_byte_scaled<0>(qu[u]), bf16_lo(x[2 * u]), acc0);
      acc1 = __fmaf_rn(e4m3_byte_scaled<1>(qu[u]), bf16_hi(x[2 * u]), acc1);
      acc0 = __fmaf_rn(e4m3_byte_scaled<2>(qu[u]), bf16_lo(x[2 * u + 1]), acc0);
      acc1 = __fmaf_rn(e4m3_byte_scaled<3>(qu[u]), bf16_hi(x[2 * u + 1]), acc1);
    }
  }
}

// 16 E4M3 codes times 16 activations held as f16 pairs, by the hardware E4M3 -> f16 conversion
// (exact: every E4M3 value is an f16 value) and mixed f16 x f16 -> fp32 FMAs (exact products).
// Elements 2i -> acc0, 2i+1 -> acc1, as in the bit-placement decode.
__device__ __forceinline__ void fp8_dot16_cvt(const uint4& q, const uint32_t* xh, float& acc0, float& acc1) {
  const uint32_t qu[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    asm("{\n\t.reg .b16 c01, c23, a0, a1, a2, a3, x0, x1, x2, x3;\n\t.reg .b32 h01, h23;\n\t"
        "mov.b32 {c01, c23}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 h01, c01;\n\t"
        "cvt.rn.f16x2.e4m3x2 h23, c23;\n\t"
        "mov.b32 {a0, a1}, h01;\n\tmov.b32 {a2, a3}, h23;\n\t"
        "mov.b32 {x0, x1}, %3;\n\tmov.b32 {x2, x3}, %4;\n\t"
        "fma.rn.f32.f16 %0, a0, x0, %0;\n\t"
        "fma.rn.f32.f16 %1, a1, x1, %1;\n\t"
        "fma.rn.f32.f16 %0, a2, x2, %0;\n\t"
        "fma.rn.f32.f16 %1, a3, x3, %1;\n\t}"
        : "+f"(acc0), "+f"(acc1)
        : "r"(qu[u]), "r"(xh[2 * u]), "r"(xh[2 * u + 1]));
  }
}

// f16 bits of v (round to nearest; exact for every BF16 value times 2^k inside the f16 range)
__device__ __forceinline__ uint32_t f32_to_f16_bits(float v) {
  unsigned short h;
  asm("cvt.rn.f16.f32 %0, %1;" : "=h"(h) : "f"(v));
  return h;
}

// Warp-uniform row value from the two per-lane accumulators (fixed tree).
template <int WT>
__device__ __forceinline__ float row_value(float acc0, float acc1, float row_scale) {
  float v = __fadd_rn(acc0, acc1);
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, m));
  if constexpr (WT == MTP_W_FP8_E4M3) v = __fmul_rn(__fmul_rn(v, kE4m3Unscale), row_scale);
  return v;
}

// Warp argmax of per-lane candidates (lowest index among equal maxima; result in every lane).
__device__ __forceinline__ ArgBest warp_arg_reduce(ArgBest b) {
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) {
    const float v = __shfl_xor_sync(0xffffffffu, b.v, m);
    const int32_t i = __shfl_xor_sync(0xffffffffu, b.i, m);
    if (i >= 0) arg_update(b, v, i);
  }
  return b;
}

// Sum over the 32 lanes of 8 per-lane partials p[0..7] (one per row), transposed: after it lane
// l holds the total of row (l >> 2) & 7. 9 shuffles instead of 40; every row's total is the same
// butterfly over lanes (pairs l^16, l^8, l^4, l^2, l^1) as a plain xor reduction, so the value
// does not depend on the row's position in the group.
__device__ __forceinline__ float transpose_reduce8(const float (&p)[8], int lane) {
  const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
  float q[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float send = b4 ? p[j] : p[j + 4];
    const float keep = b4 ? p[j + 4] : p[j];
    q[j] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, 16));
  }
  float r[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const float send = b3 ? q[j] : q[j + 2];
    const float keep = b3 ? q[j + 2] : q[j];
    r[j] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, 8));
  }
  const float send = b2 ? r[0] : r[1];
  const float keep = b2 ? r[1] : r[0];
  float v = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, 4));
  v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 2));
  v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 1));
  return v;
}

template <int WT>
using XhatLayout = typename std::conditional<WT == MTP_W_BF16, LayoutIdentity, LayoutFp8>::type;

template <int NT, class Layout>
__device__ void final_norm_prologue(const SweepArgs& a, int nb, uint16_t* vec, int vec_elems,
                                    float* red) {
  auto job = [&](int b) {
    return NormJob{a.x + static_cast<size_t>(b) * a.H, a.final_norm_w,
                   vec + static_cast<size_t>(b) * vec_elems, true};
  };
  rms_norm_multi_to_smem<NT>(nb, a.H, a.inv_h, a.eps, red, job, Layout{});
  __syncthreads();
}

// ------------------------------------------------------------------------------------------
// B = 1, H = NVL * 32 * (elements per 16-byte vector): xhat in registers, one row per stage,
// rows reduced eight at a time (the per-row partial goes to slot i % 8 by selects, the row loop
// stays rolled). NWR warps per CTA. For FP8 with kCvt the codes go through the hardware
// E4M3 -> f16 conversion and xhat is held as f16 scaled by 2^k (k chosen from max |xhat| so that
// the largest value lands in [2^14, 2^15)); the row sum is scaled back by 2^-k. Products stay
// exact and the sums are the bit-placement sums scaled by a power of two, so both decodes give
// the same logits (activations below 2^-31 max |xhat| excepted).
// ------------------------------------------------------------------------------------------
constexpr int kGroup = 8;

template <int WT, int NVL, int NWR, bool kMixed, bool kCvt>
__device__ __forceinline__ void sweep_regx_body(const SweepArgs& a, const HostBack* hb) {
  constexpr int EB = (WT == MTP_W_BF16) ? 2 : 1;
  constexpr int EPV = 16 / EB;
  constexpr int H = NVL * 32 * EPV;
  constexpr uint32_t RB = static_cast<uint32_t>(H) * EB;  // row bytes
  constexpr int XW = EPV / 2;                             // activation pairs per vector
  constexpr bool kF16 = (WT == MTP_W_FP8_E4M3) && kCvt;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ float xmax_s[NWR];

  const int S = a.stages;
  const int64_t V = a.V;
  uint8_t* stages = smem;
  uint16_t* vec = reinterpret_cast<uint16_t*>(stages + static_cast<size_t>(NWR) * S * RB);
  uint64_t* bars = reinterpret_cast<uint64_t*>(vec + H);
  float* red = reinterpret_cast<float*>(bars + NWR * S);
  ArgBest* wbest = reinterpret_cast<ArgBest*>(red + kRedBytes / sizeof(float));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // per-warp queues: row and row scale of each stage, row and scale of each group slot
  int* rowq = reinterpret_cast<int*>(wbest + kWarps * kMaxB) + warp * (2 * kMaxStages + 2 * kGroup);
  float* scq = reinterpret_cast<float*>(rowq + kMaxStages);
  int* grow = rowq + 2 * kMaxStages;
  float* gsc = reinterpret_cast<float*>(grow + kGroup);
  // Rows are handed out dynamically: each warp's first S rows are fixed (they are prefetched
  // before the preceding kernel has finished), the rest are claimed kClaim at a time from a
  // counter in the workspace header. With a fixed split, CTAs ended their last rows up to
  // ~60 us apart (some SMs draw less bandwidth) and the kernel waited for the slowest.
  constexpr int kClaim = (WT == MTP_W_BF16) ? 4 : 8;  // ~48 KB of weights per claim
  unsigned int* row_counter = reinterpret_cast<unsigned int*>(a.ws + kRowCounterOffset);
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * NWR + warp;
  const int64_t nstatic = V < static_cast<int64_t>(gridDim.x) * NWR * S ? V : static_cast<int64_t>(gridDim.x) * NWR * S;
  // issue side, lane 0 only: current block [cur, cur_end) and the block claimed ahead
  int64_t cur = gw * S, cur_end = cur + S < V ? cur + S : V;
  unsigned int nxt = 0;
  bool have_nxt = false, exhausted = false;
  int issued = 0;
  float pend_scale = 1.0f;
  int pend_stage = -1;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NWR * S; ++i) mbar_init(smem_addr(&bars[i]), 1);
    fence_barrier_init();
  }
  __syncthreads();

  uint8_t* my_stages = stages + static_cast<size_t>(warp) * S * RB;
  uint64_t* my_bars = bars + warp * S;
  const uint64_t policy = l2_evict_first_policy();
  int ps = 0;
  auto issue_next = [&]() {  // lane 0
    if (cur >= cur_end) {
      if (!have_nxt) {
        exhausted = true;
        return;
      }
      cur = nstatic + static_cast<int64_t>(nxt);
      cur_end = cur + kClaim < V ? cur + kClaim : V;
      if (cur >= V) {
        exhausted = true;
        have_nxt = false;
        return;
      }
      nxt = atomicAdd(row_counter, static_cast<unsigned int>(kClaim));  // the one after, ahead of need
    }
    const int64_t row = cur++;
    const uint32_t bar = smem_addr(&my_bars[ps]);
    mbar_arrive_expect_tx(bar, RB);
    bulk_copy_g2s(smem_addr(my_stages + static_cast<size_t>(ps) * RB), a.W + row * RB, RB, bar, policy);
    rowq[ps] = static_cast<int>(row);
    if constexpr (WT == MTP_W_FP8_E4M3) {
      // the scale load is stored one issue later, when it has long arrived
      if (pend_stage >= 0) scq[pend_stage] = pend_scale;
      pend_scale = __ldg(a.scale + row);
      pend_stage = ps;
    }
    ++issued;
    if (++ps == S) ps = 0;
  };
  auto flush_scale = [&]() {  // lane 0
    if constexpr (WT == MTP_W_FP8_E4M3) {
      if (pend_stage >= 0) scq[pend_stage] = pend_scale;
      pend_stage = -1;
    }
  };
  if (lane == 0) {
    for (int t = 0; t < S && !exhausted; ++t) issue_next();
    if (exhausted) flush_scale();  // only when V leaves nothing to claim
  }

  pdl_wait_prior_grid();  // x comes from the preceding kernel; the row counter is free again
  if (lane == 0 && nstatic < V) {
    nxt = atomicAdd(row_counter, static_cast<unsigned int>(kClaim));
    have_nxt = true;
  }
  final_norm_prologue<NWR * 32, XhatLayout<WT>>(a, 1, vec, H, red);
  float unscale = 1.0f;  // 2^-k for the f16 activations
  float xscale = 1.0f;   // 2^k
  if constexpr (kF16) {
    float m = 0.0f;
    for (int k = threadIdx.x; k < H; k += NWR * 32) m = fmaxf(m, fabsf(bf16_bits_to_f32(vec[k])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) xmax_s[warp] = m;
    __syncthreads();
    m = xmax_s[0];
    for (int w = 1; w < NWR; ++w) m = fmaxf(m, xmax_s[w]);
    int e = 0;
    const bool finite_pos = m > 0.0f && m <= 3.0e38f;
    if (finite_pos) (void)frexpf(m, &e);  // m in [2^(e-1), 2^e)
    const int k = finite_pos ? 15 - e : 0;
    xscale = ldexpf(1.0f, k);
    unscale = ldexpf(1.0f, -k);
  }
  uint32_t xr[NVL][XW];
#pragma unroll
  for (int t = 0; t < NVL; ++t) {
    const uint4* xv = reinterpret_cast<const uint4*>(vec);
    if constexpr (WT == MTP_W_BF16) {
      const uint4 q = xv[t * 32 + lane];
      xr[t][0] = q.x; xr[t][1] = q.y; xr[t][2] = q.z; xr[t][3] = q.w;
    } else {
      const uint4 q0 = xv[t * 64 + lane], q1 = xv[t * 64 + 32 + lane];  // LayoutFp8 slots
      const uint32_t u[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
      for (int p = 0; p < 8; ++p) {
        if constexpr (kF16) {
          xr[t][p] = f32_to_f16_bits(__fmul_rn(bf16_lo(u[p]), xscale)) |
                     (f32_to_f16_bits(__fmul_rn(bf16_hi(u[p]), xscale)) << 16);
        } else {
          xr[t][p] = u[p];
        }
      }
    }
  }
  pdl_launch_dependents();

  ArgBest best{0.0f, -1};
  const int my_slot = (lane >> 2) & 7;  // row of a group whose total this lane ends up with
  float part[kGroup];
#pragma unroll
  for (int j = 0; j < kGroup; ++j) part[j] = 0.0f;
  int cs = 0, i_fail = -1, consumed = 0;
  uint32_t parity = 0;
  int n_issued = __shfl_sync(0xffffffffu, issued, 0);
#pragma unroll 1
  while (consumed < n_issued) {
    const int jj = consumed & (kGroup - 1);
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_addr(&my_bars[cs]), parity, a.wait_ns))) {
      i_fail = consumed;
      break;
    }
    const uint4* wv = reinterpret_cast<const uint4*>(my_stages + static_cast<size_t>(cs) * RB);
    float acc0 = 0.0f, acc1 = 0.0f;
#pragma unroll
    for (int t = 0; t < NVL; ++t) {
      const uint4 q = wv[t * 32 + lane];
      if constexpr (WT == MTP_W_BF16) {
        fma_pair<kMixed>(acc0, acc1, q.x, xr[t][0]);
        fma_pair<kMixed>(acc0, acc1, q.y, xr[t][1]);
        fma_pair<kMixed>(acc0, acc1, q.z, xr[t][2]);
        fma_pair<kMixed>(acc0, acc1, q.w, xr[t][3]);
      } else if constexpr (kF16) {
        fp8_dot16_cvt(q, xr[t], acc0, acc1);
      } else {
        fp8_dot16<kMixed>(q, xr[t], acc0, acc1);
      }
    }
    const float pv = __fadd_rn(acc0, acc1);
#pragma unroll
    for (int j = 0; j < kGroup; ++j) part[j] = (j == jj) ? pv : part[j];
    if (lane == 0) {
      grow[jj] = rowq[cs];
      if constexpr (WT == MTP_W_FP8_E4M3) gsc[jj] = scq[cs];
    }
    __syncwarp();
    ++consumed;
    if (lane == 0 && !exhausted) {
      fence_proxy_async_smem();
      issue_next();
      if (exhausted) flush_scale();
    }
    n_issued = __shfl_sync(0xffffffffu, issued, 0);
    if (++cs == S) { cs = 0; parity ^= 1u; }
    if (jj == kGroup - 1 || consumed == n_issued) {
      __syncwarp();
      float v = transpose_reduce8(part, lane);
      if (my_slot <= jj) {
        const int my_row = grow[my_slot];
        if constexpr (kF16) v = __fmul_rn(__fmul_rn(v, unscale), gsc[my_slot]);
        else if constexpr (WT == MTP_W_FP8_E4M3) v = __fmul_rn(__fmul_rn(v, kE4m3Unscale), gsc[my_slot]);
        if ((lane & 3) == 0 && a.logits != nullptr) a.logits[my_row] = v;
        arg_update(best, v, static_cast<int32_t>(my_row));
      }
#pragma unroll
      for (int j = 0; j < kGroup; ++j) part[j] = 0.0f;
      __syncwarp();
    }
  }
  if (i_fail >= 0) {
    if (lane == 0) {
      store_status(a.status, MTP_ERR_TIMEOUT);
      // let the copies still in flight land before the CTA's shared memory is released
      int s2 = cs;
      uint32_t par = parity;
      for (int u = i_fail; u < n_issued && u < i_fail + S; ++u) {
        (void)mbar_wait_bounded(smem_addr(&my_bars[s2]), par);
        if (++s2 == S) { s2 = 0; par ^= 1u; }
      }
    }
  }
  __syncwarp();
  best = warp_arg_reduce(best);
  argmax_finish<1>(&best, 1, wbest, a, hb);
}

template <int WT, int NVL, int NWR, bool kMixed, bool kCvt>
__global__ void __launch_bounds__(NWR * 32, 1) sweep_regx_kernel(const SweepArgs a) {
  sweep_regx_body<WT, NVL, NWR, kMixed, kCvt>(a, nullptr);
}

// The same for a recorded host-buffer step (HostBack).
template <int WT, int NVL, int NWR, bool kMixed, bool kCvt>
__global__ void __launch_bounds__(NWR * 32, 1) sweep_regx_hb_kernel(const SweepArgs a, const HostBack hb) {
  sweep_regx_body<WT, NVL, NWR, kMixed, kCvt>(a, &hb);
}

// ------------------------------------------------------------------------------------------
// B <= 4 sequences, H * sizeof(weight) a multiple of 16: xhat in shared memory, 4 KB stages.
// ------------------------------------------------------------------------------------------
template <int WT, int NB, bool kMixed>
__global__ void __launch_bounds__(kThreads, 1) sweep_tma_kernel(const SweepArgs a) {
  constexpr int EB = (WT == MTP_W_BF16) ? 2 : 1;  // bytes per weight element
  constexpr int EPV = 16 / EB;                    // weight elements per 16-byte vector
  constexpr int NW = kWarps;
  extern __shared__ __align__(128) uint8_t smem[];

  const int S = a.stages;
  const int H = a.H;
  const int64_t V = a.V;
  const int64_t row_bytes = static_cast<int64_t>(H) * EB;
  const int cpr = static_cast<int>((row_bytes + kChunk - 1) / kChunk);  // chunks per row
  const uint32_t last_bytes = static_cast<uint32_t>(row_bytes - static_cast<int64_t>(cpr - 1) * kChunk);
  const int vec_elems = ((H / EPV + 31) / 32) * 32 * EPV;

  uint8_t* stages = smem;
  uint16_t* vec = reinterpret_cast<uint16_t*>(stages + static_cast<size_t>(NW) * S * kChunk);
  uint64_t* bars = reinterpret_cast<uint64_t*>(vec + static_cast<size_t>(NB) * vec_elems);
  float* red = reinterpret_cast<float*>(bars + NW * S);
  ArgBest* wbest = reinterpret_cast<ArgBest*>(red + kRedBytes / sizeof(float));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t r0 = V * blockIdx.x / gridDim.x;
  const int64_t r1 = V * (blockIdx.x + 1) / gridDim.x;
  const int64_t cta_rows = r1 - r0;
  const int nrows = cta_rows > warp ? static_cast<int>((cta_rows - warp + NW - 1) / NW) : 0;
  const int nitems = nrows * cpr;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NW * S; ++i) mbar_init(smem_addr(&bars[i]), 1);
    fence_barrier_init();
  }
  __syncthreads();

  uint8_t* my_stages = stages + static_cast<size_t>(warp) * S * kChunk;
  uint64_t* my_bars = bars + warp * S;
  const uint64_t policy = l2_evict_first_policy();
  int pi = 0, pc = 0, ps = 0;  // producer cursor (lane 0 only): row, chunk, stage
  auto issue_next = [&]() {
    const int64_t row = r0 + warp + static_cast<int64_t>(pi) * NW;
    const uint32_t bytes = (pc == cpr - 1) ? last_bytes : static_cast<uint32_t>(kChunk);
    const uint8_t* src = a.W + row * row_bytes + static_cast<int64_t>(pc) * kChunk;
    const uint32_t bar = smem_addr(&my_bars[ps]);
    mbar_arrive_expect_tx(bar, bytes);
    bulk_copy_g2s(smem_addr(my_stages + static_cast<size_t>(ps) * kChunk), src, bytes, bar, policy);
    if (++pc == cpr) { pc = 0; ++pi; }
    if (++ps == S) ps = 0;
  };
  const int prefill = nitems < S ? nitems : S;
  if (lane == 0)
    for (int t = 0; t < prefill; ++t) issue_next();

  pdl_wait_prior_grid();  // x comes from the preceding kernel
  final_norm_prologue<kThreads, XhatLayout<WT>>(a, NB, vec, vec_elems, red);
  pdl_launch_dependents();

  float acc[NB][2];
#pragma unroll
  for (int b = 0; b < NB; ++b) acc[b][0] = acc[b][1] = 0.0f;
  ArgBest best[NB];
#pragma unroll
  for (int b = 0; b < NB; ++b) best[b] = ArgBest{0.0f, -1};

  int ci = 0, cc = 0, cs = 0, t_fail = -1;  // consumer cursor: row, chunk, stage
  uint32_t parity = 0;
  float row_scale = 1.0f;
  for (int t = 0; t < nitems; ++t) {
    const int64_t row = r0 + warp + static_cast<int64_t>(ci) * NW;
    if constexpr (WT == MTP_W_FP8_E4M3) {
      if (cc == 0) row_scale = __ldg(a.scale + row);
    }
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_addr(&my_bars[cs]), parity, a.wait_ns))) {
      t_fail = t;
      break;
    }
    const uint4* wv = reinterpret_cast<const uint4*>(my_stages + static_cast<size_t>(cs) * kChunk);
    const int nv = static_cast<int>(((cc == cpr - 1) ? last_bytes : static_cast<uint32_t>(kChunk)) >> 4);
    const int J0 = cc * (kChunk / 16);
#pragma unroll 4
    for (int j = lane; j < nv; j += 32) {
      const uint4 q = wv[j];
      const int J = J0 + j;
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        const uint4* xb = reinterpret_cast<const uint4*>(vec + static_cast<size_t>(b) * vec_elems);
        if constexpr (WT == MTP_W_BF16) {
          const uint4 xq = xb[J];
          fma_pair<kMixed>(acc[b][0], acc[b][1], q.x, xq.x);
          fma_pair<kMixed>(acc[b][0], acc[b][1], q.y, xq.y);
          fma_pair<kMixed>(acc[b][0], acc[b][1], q.z, xq.z);
          fma_pair<kMixed>(acc[b][0], acc[b][1], q.w, xq.w);
        } else {
          const int slot0 = (J >> 5) * 64 + (J & 31);  // LayoutFp8 slots of vector J
          const uint4 x0 = xb[slot0], x1 = xb[slot0 + 32];
          const uint32_t xu[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
          fp8_dot16<kMixed>(q, xu, acc[b][0], acc[b][1]);
        }
      }
    }
    __syncwarp();
    if (lane == 0 && t + S < nitems) {
      fence_proxy_async_smem();
      issue_next();
    }
    if (++cs == S) { cs = 0; parity ^= 1u; }
    if (++cc == cpr) {
      cc = 0;
      ++ci;
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        const float v = row_value<WT>(acc[b][0], acc[b][1], row_scale);
        if (lane == 0 && a.logits != nullptr) a.logits[static_cast<int64_t>(b) * V + row] = v;
        arg_update(best[b], v, static_cast<int32_t>(row));
        acc[b][0] = acc[b][1] = 0.0f;
      }
    }
  }
  if (t_fail >= 0 && lane == 0) {
    store_status(a.status, MTP_ERR_TIMEOUT);
    // let the copies still in flight land before the CTA's shared memory is released
    int s = cs;
    uint32_t par = parity;
    for (int u = t_fail; u < nitems && u < t_fail + S; ++u) {
      (void)mbar_wait_bounded(smem_addr(&my_bars[s]), par);
      if (++s == S) { s = 0; par ^= 1u; }
    }
  }
  __syncwarp();
  argmax_finish<NB>(best, NB, wbest, a);
}

// ------------------------------------------------------------------------------------------
// Plain-load sweep for any H (rows not 16-byte aligned) and any B <= 16: one warp per row,
// lanes striding over k. Same numerics (fp32 products and sums, fixed order per row).
// ------------------------------------------------------------------------------------------
template <int WT>
__global__ void __launch_bounds__(kThreads) sweep_plain_kernel(const SweepArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int H = a.H, nb = a.B;
  const int64_t V = a.V;
  uint16_t* vec = reinterpret_cast<uint16_t*>(smem);
  const int vec_elems = ((H + 7) / 8) * 8;
  float* red = reinterpret_cast<float*>(vec + static_cast<size_t>(nb) * vec_elems);
  ArgBest* wbest = reinterpret_cast<ArgBest*>(red + kRedBytes / sizeof(float));

  pdl_wait_prior_grid();
  final_norm_prologue<kThreads, LayoutIdentity>(a, nb, vec, vec_elems, red);
  pdl_launch_dependents();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  ArgBest best[kMaxB];
  for (int b = 0; b < kMaxB; ++b) best[b] = ArgBest{0.0f, -1};
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
  const int64_t tw = static_cast<int64_t>(gridDim.x) * kWarps;
  for (int64_t row = gw; row < V; row += tw) {
    float scale = 1.0f;
    if constexpr (WT == MTP_W_FP8_E4M3) scale = __ldg(a.scale + row);
    for (int b = 0; b < nb; ++b) {
      float acc = 0.0f;
      const uint16_t* xb = vec + static_cast<size_t>(b) * vec_elems;
      for (int k = lane; k < H; k += 32) {
        float wv;
        if constexpr (WT == MTP_W_BF16) {
          wv = bf16_bits_to_f32(reinterpret_cast<const uint16_t*>(a.W)[row * H + k]);
        } else {
          wv = e4m3_byte_scaled<0>(a.W[row * H + k]);
        }
        acc = __fmaf_rn(wv, bf16_bits_to_f32(xb[k]), acc);
      }
      for (int m = 16; m > 0; m >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, m));
      if constexpr (WT == MTP_W_FP8_E4M3) acc = __fmul_rn(__fmul_rn(acc, kE4m3Unscale), scale);
      if (lane == 0 && a.logits != nullptr) a.logits[static_cast<int64_t>(b) * V + row] = acc;
      arg_update(best[b], acc, static_cast<int32_t>(row));
    }
  }
  argmax_finish<kMaxB>(best, nb, wbest, a);
}

cudaError_t launch_sweep_kernel(void (*kernel)(SweepArgs), unsigned grid, unsigned threads, size_t smem,
                                cudaStream_t stream, SweepArgs a) {
  void* args[] = {&a};
  return launch_pdl(reinterpret_cast<const void*>(kernel), dim3(grid), dim3(threads), smem, stream, args);
}

constexpr bool kMixedDefault = MTP_MIXED_FMA != 0;
// per-warp row queues of the single-sequence kernel (up to 16 warps)
constexpr size_t kQueueBytes = static_cast<size_t>(16) * (2 * kMaxStages + 2 * kGroup) * 4;
constexpr size_t kMisc = kRedBytes + static_cast<size_t>(kWarps) * kMaxB * sizeof(ArgBest) + kQueueBytes + 256;

template <int WT, int NB>
cudaError_t launch_tma(SweepArgs a, const DeviceInfo& di, unsigned grid, size_t fixed, cudaStream_t stream) {
  const size_t per_stage = static_cast<size_t>(kWarps) * (kChunk + 8);
  int S = static_cast<int>((static_cast<size_t>(di.smem_optin) - fixed) / per_stage);
  if (S > kMaxStages) S = kMaxStages;
  a.stages = S;
  return launch_sweep_kernel(sweep_tma_kernel<WT, NB, kMixedDefault>, grid, kThreads, fixed + S * per_stage,
                             stream, a);
}

#ifndef MTP_REGX_WARPS_BF16
#define MTP_REGX_WARPS_BF16 8
#endif
#ifndef MTP_REGX_WARPS_FP8
#define MTP_REGX_WARPS_FP8 12
#endif
#ifndef MTP_FP8_CVT
#define MTP_FP8_CVT 1
#endif

// B = 1 register-xhat kernel, if this H has an instantiation and the stages fit; with hb, the
// kernel that also hands the result back to host memory.
template <int WT>
cudaError_t try_launch_regx(SweepArgs a, const DeviceInfo& di, unsigned grid, cudaStream_t stream,
                            bool* launched, const HostBack* hb = nullptr) {
  constexpr int EB = (WT == MTP_W_BF16) ? 2 : 1;
  constexpr int EPV = 16 / EB;
  constexpr int NWR = (WT == MTP_W_BF16) ? MTP_REGX_WARPS_BF16 : MTP_REGX_WARPS_FP8;
  constexpr bool kCvt = MTP_FP8_CVT != 0;
  *launched = false;
  if (!MTP_REGX || a.H % (32 * EPV) != 0) return cudaSuccess;
  const int nvl = a.H / (32 * EPV);
  void (*k)(SweepArgs) = nullptr;
  void (*khb)(SweepArgs, HostBack) = nullptr;
  if constexpr (WT == MTP_W_BF16) {
    switch (nvl) {
      case 16:  // H = 4096
        k = sweep_regx_kernel<WT, 16, NWR, kMixedDefault, kCvt>;
        khb = sweep_regx_hb_kernel<WT, 16, NWR, kMixedDefault, kCvt>;
        break;
      case 24:  // H = 6144
        k = sweep_regx_kernel<WT, 24, NWR, kMixedDefault, kCvt>;
        khb = sweep_regx_hb_kernel<WT, 24, NWR, kMixedDefault, kCvt>;
        break;
      case 28:  // H = 7168
        k = sweep_regx_kernel<WT, 28, NWR, kMixedDefault, kCvt>;
        khb = sweep_regx_hb_kernel<WT, 28, NWR, kMixedDefault, kCvt>;
        break;
      default: return cudaSuccess;
    }
  } else {
    switch (nvl) {
      case 8:  // H = 4096
        k = sweep_regx_kernel<WT, 8, NWR, kMixedDefault, kCvt>;
        khb = sweep_regx_hb_kernel<WT, 8, NWR, kMixedDefault, kCvt>;
        break;
      case 12:  // H = 6144
        k = sweep_regx_kernel<WT, 12, NWR, kMixedDefault, kCvt>;
        khb = sweep_regx_hb_kernel<WT, 12, NWR, kMixedDefault, kCvt>;
        break;
      case 14:  // H = 7168
        k = sweep_regx_kernel<WT, 14, NWR, kMixedDefault, kCvt>;
        khb = sweep_regx_hb_kernel<WT, 14, NWR, kMixedDefault, kCvt>;
        break;
      default: return cudaSuccess;
    }
  }
  const size_t rb = static_cast<size_t>(a.H) * EB;
  const size_t fixed = static_cast<size_t>(a.H) * 2 + kMisc;
  const size_t per_stage = static_cast<size_t>(NWR) * (rb + 8);
  if (fixed + 2 * per_stage > static_cast<size_t>(di.smem_optin)) return cudaSuccess;
  int S = static_cast<int>((static_cast<size_t>(di.smem_optin) - fixed) / per_stage);
  if (S > kMaxStages) S = kMaxStages;
  a.stages = S;
  *launched = true;
  if (hb != nullptr) {
    HostBack h = *hb;
    void* args[] = {&a, &h};
    return launch_pdl(reinterpret_cast<const void*>(khb), dim3(grid), dim3(NWR * 32), fixed + S * per_stage, stream,
                      args);
  }
  return launch_sweep_kernel(k, grid, NWR * 32, fixed + S * per_stage, stream, a);
}

}  // namespace

size_t sweep_workspace_bytes(int /*B*/) { return static_cast<size_t>(kWsBytes); }

cudaError_t launch_sweep_handback(const SweepArgs& in, const HostBack& hb, cudaStream_t stream, bool* done) {
  *done = false;
  DeviceInfo di;
  cudaError_t err = device_info(&di);
  if (err != cudaSuccess) return err;
  const int EB = (in.w_dtype == MTP_W_BF16) ? 2 : 1;
  if (in.B != 1 || (static_cast<int64_t>(in.H) * EB) % 16 != 0) return cudaSuccess;
  const int64_t want = (static_cast<int64_t>(in.V) + kWarps - 1) / kWarps;
  int64_t g = di.sm_count < want ? di.sm_count : want;
  if (g > kMaxGrid) g = kMaxGrid;
  if (g < 1) g = 1;
  return in.w_dtype == MTP_W_BF16 ? try_launch_regx<MTP_W_BF16>(in, di, static_cast<unsigned>(g), stream, done, &hb)
                                  : try_launch_regx<MTP_W_FP8_E4M3>(in, di, static_cast<unsigned>(g), stream, done, &hb);
}

cudaError_t launch_sweep(const SweepArgs& in, cudaStream_t stream) {
  DeviceInfo di;
  cudaError_t err = device_info(&di);
  if (err != cudaSuccess) return err;
  SweepArgs a = in;
  const int EB = (a.w_dtype == MTP_W_BF16) ? 2 : 1;
  const int EPV = 16 / EB;
  const bool rows16 = (static_cast<int64_t>(a.H) * EB) % 16 == 0;
  const int64_t want = (static_cast<int64_t>(a.V) + kWarps - 1) / kWarps;
  int64_t g = di.sm_count < want ? di.sm_count : want;
  if (g > kMaxGrid) g = kMaxGrid;
  if (g < 1) g = 1;
  const unsigned grid = static_cast<unsigned>(g);
  if (rows16 && a.B == 1) {
    bool launched = false;
    err = (a.w_dtype == MTP_W_BF16) ? try_launch_regx<MTP_W_BF16>(a, di, grid, stream, &launched)
                                    : try_launch_regx<MTP_W_FP8_E4M3>(a, di, grid, stream, &launched);
    if (launched || err != cudaSuccess) return err;
  }
  if (a.B >= MTP_TC_MIN_B) {
    bool launched = false;
    err = launch_sweep_tc(a, stream, &launched);
    if (launched || err != cudaSuccess) return err;
  }
  if (rows16 && a.B <= kTmaMaxB) {
    const int vec_elems = ((a.H / EPV + 31) / 32) * 32 * EPV;
    const size_t fixed = static_cast<size_t>(a.B) * vec_elems * 2 + kMisc;
    const size_t per_stage = static_cast<size_t>(kWarps) * (kChunk + 8);
    if (fixed + 2 * per_stage <= static_cast<size_t>(di.smem_optin)) {
      if (a.w_dtype == MTP_W_BF16) {
        switch (a.B) {
          case 1: return launch_tma<MTP_W_BF16, 1>(a, di, grid, fixed, stream);
          case 2: return launch_tma<MTP_W_BF16, 2>(a, di, grid, fixed, stream);
          case 3: return launch_tma<MTP_W_BF16, 3>(a, di, grid, fixed, stream);
          default: return launch_tma<MTP_W_BF16, 4>(a, di, grid, fixed, stream);
        }
      } else {
        switch (a.B) {
          case 1: return launch_tma<MTP_W_FP8_E4M3, 1>(a, di, grid, fixed, stream);
          case 2: return launch_tma<MTP_W_FP8_E4M3, 2>(a, di, grid, fixed, stream);
          case 3: return launch_tma<MTP_W_FP8_E4M3, 3>(a, di, grid, fixed, stream);
          default: return launch_tma<MTP_W_FP8_E4M3, 4>(a, di, grid, fixed, stream);
        }
      }
    }
  }
  const int vec_elems = ((a.H + 7) / 8) * 8;
  const size_t smem = static_cast<size_t>(a.B) * vec_elems * 2 + kMisc;
  if (smem > static_cast<size_t>(di.smem_optin)) return cudaErrorNotSupported;
  a.stages = 0;
  if (a.w_dtype == MTP_W_BF16)
    return launch_sweep_kernel(sweep_plain_kernel<MTP_W_BF16>, grid, kThreads, smem, stream, a);
  return launch_sweep_kernel(sweep_plain_kernel<MTP_W_FP8_E4M3>, grid, kThreads, smem, stream, a);
}

}  // namespace mtp
