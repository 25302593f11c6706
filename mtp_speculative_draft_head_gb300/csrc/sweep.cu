// Output stage of the MTP draft head: shared_head.norm, the lm_head vocabulary sweep and the
// argmax, fused into one kernel ("glm5next_mtp_head.rs", `forward_one`: `norm` of x with
// final_norm in place, `dense_gemv` / `dense_gemv_fp8w` over the vocabulary, `argmax_bf16`).
//
// Design (one GB300, HBM-bound GEMV, no tensor cores at this batch size):
//  * Persistent grid: one 256-thread CTA per SM, each owning a contiguous range of vocabulary
//    rows (V split evenly, so the tail is at most one row per CTA).
//  * Each warp streams its own rows through a private ring of shared-memory stages filled by
//    1-D bulk async copies (TMA engine, `cp.async.bulk` + mbarrier transaction counts, L2
//    evict-first). The weight stream never touches registers before shared memory, so a few
//    warps keep ~100-200 KB per SM in flight.
//  * Before waiting for the preceding kernel (programmatic dependent launch) each warp already
//    issues its first stages: the weights do not depend on x.
//  * Prologue: every CTA computes xhat = rms_norm_vanilla(x, final_norm_w) for its B sequences
//    into shared memory (BF16, laid out so the per-lane reads are bank-conflict free).
//  * Each row is reduced by one warp with a fixed lane->element map and a fixed shuffle tree,
//    so identical rows give bit-identical logits (exact ties stay exact).
//  * Epilogue: FP32 logits written once (optional), a per-warp then per-CTA (max, lowest index)
//    and a last-CTA-done combine of the per-CTA partials into draft[b]. No CTA ever waits for
//    another; the counter returns itself to zero for the next call or graph replay.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

namespace mtp {

namespace {

// ------------------------------------------------------------------------------------------
// Per-CTA epilogue: combine warp bests, publish the CTA partial, and let the last CTA finish.
// best[] is uniform across the lanes of a warp.
// ------------------------------------------------------------------------------------------
template <int NB>
__device__ void argmax_finish(const ArgBest* best, int nb, ArgBest* wbest, uint8_t* ws,
                              int32_t* draft) {
  __shared__ int is_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  if (lane == 0) {
#pragma unroll
    for (int b = 0; b < NB; ++b)
      if (b < nb) wbest[warp * nb + b] = best[b];
  }
  __syncthreads();
  ArgBest* part = reinterpret_cast<ArgBest*>(ws + kWsHeader);
  unsigned int* counter = reinterpret_cast<unsigned int*>(ws);
  if (threadIdx.x < nb) {
    ArgBest c{0.0f, -1};
    for (int w = 0; w < nwarps; ++w) {
      const ArgBest o = wbest[w * nb + threadIdx.x];
      if (o.i >= 0) arg_update(c, o.v, o.i);
    }
    part[blockIdx.x * nb + threadIdx.x] = c;
    __threadfence();
  }
  __syncthreads();
  if (threadIdx.x == 0) is_last = (atomicAdd(counter, 1u) == gridDim.x - 1) ? 1 : 0;
  __syncthreads();
  if (is_last) {
    __threadfence();
    if (threadIdx.x < nb) {
      ArgBest c{0.0f, -1};
      for (unsigned int g = 0; g < gridDim.x; ++g) {
        const uint2 raw = __ldcg(reinterpret_cast<const uint2*>(part + g * nb + threadIdx.x));
        const ArgBest o{__uint_as_float(raw.x), static_cast<int32_t>(raw.y)};
        if (o.i >= 0) arg_update(c, o.v, o.i);
      }
      draft[threadIdx.x] = c.i;
    }
    if (threadIdx.x == 0) atomicExch(counter, 0u);
  }
}

// Mixed-precision FMA: fp32 accumulator += bf16 * bf16 (both halves of 32-bit pairs).
__device__ __forceinline__ void fma2_bf16(float& acc0, float& acc1, uint32_t w, uint32_t x) {
  asm("{\n\t.reg .b16 wl, wh, xl, xh;\n\t"
      "mov.b32 {wl, wh}, %2;\n\t"
      "mov.b32 {xl, xh}, %3;\n\t"
      "fma.rn.f32.bf16 %0, wl, xl, %0;\n\t"
      "fma.rn.f32.bf16 %1, wh, xh, %1;\n\t}"
      : "+f"(acc0), "+f"(acc1)
      : "r"(w), "r"(x));
}

// Four E4M3 codes -> two BF16 pairs holding value * 2^-120 (sign to bit 15, magnitude bits
// EEEE.MMM to bits 10..4 of each half: BF16 exponent field 0000EEEE, mantissa MMM0000).
__device__ __forceinline__ void e4m3x4_to_bf16x2x2(uint32_t w, uint32_t& p01, uint32_t& p23) {
  const uint32_t m = w & 0x7F7F7F7Fu;
  const uint32_t s = w & 0x80808080u;
  p01 = __byte_perm(m, 0u, 0x4140u) * 16u + __byte_perm(s, 0u, 0x1404u);
  p23 = __byte_perm(m, 0u, 0x4342u) * 16u + __byte_perm(s, 0u, 0x3424u);
}

// ------------------------------------------------------------------------------------------
// TMA-pipelined sweep, B <= 4 sequences, H * sizeof(weight) a multiple of 16.
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
  ArgBest* wbest = reinterpret_cast<ArgBest*>(red + 2 * NW + 2);

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
  // producer cursor (lane 0 only)
  int pi = 0, pc = 0, ps = 0;
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

  // x is produced by the preceding kernel: wait for it only now.
  pdl_wait_prior_grid();
  for (int b = 0; b < NB; ++b) {
    if constexpr (WT == MTP_W_BF16)
      rms_norm_to_smem<kThreads>(a.x + static_cast<size_t>(b) * H, a.final_norm_w, H, a.eps,
                                 vec + static_cast<size_t>(b) * vec_elems, red, true, LayoutIdentity{});
    else
      rms_norm_to_smem<kThreads>(a.x + static_cast<size_t>(b) * H, a.final_norm_w, H, a.eps,
                                 vec + static_cast<size_t>(b) * vec_elems, red, true, LayoutFp8{});
    __syncthreads();
  }
  pdl_launch_dependents();

  float acc[NB][2];
#pragma unroll
  for (int b = 0; b < NB; ++b) acc[b][0] = acc[b][1] = 0.0f;
  ArgBest best[NB];
#pragma unroll
  for (int b = 0; b < NB; ++b) best[b] = ArgBest{0.0f, -1};

  int ci = 0, cc = 0, cs = 0;  // consumer cursor: row, chunk, stage
  uint32_t parity = 0;
  float row_scale = 1.0f;
  int t_fail = -1;
  for (int t = 0; t < nitems; ++t) {
    const int64_t row = r0 + warp + static_cast<int64_t>(ci) * NW;
    if constexpr (WT == MTP_W_FP8_E4M3) {
      if (cc == 0) row_scale = __ldg(a.scale + row);
    }
    const uint32_t bar = smem_addr(&my_bars[cs]);
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(bar, parity))) {
      t_fail = t;
      break;
    }
    const uint8_t* st = my_stages + static_cast<size_t>(cs) * kChunk;
    const int nv = static_cast<int>(((cc == cpr - 1) ? last_bytes : static_cast<uint32_t>(kChunk)) >> 4);
    const int J0 = cc * (kChunk / 16);
    const uint4* wv = reinterpret_cast<const uint4*>(st);
#pragma unroll 4
    for (int j = lane; j < nv; j += 32) {
      const uint4 q = wv[j];
      const int J = J0 + j;
      if constexpr (WT == MTP_W_BF16) {
        if constexpr (kMixed) {
#pragma unroll
          for (int b = 0; b < NB; ++b) {
            const uint4 xq = reinterpret_cast<const uint4*>(vec + static_cast<size_t>(b) * vec_elems)[J];
            fma2_bf16(acc[b][0], acc[b][1], q.x, xq.x);
            fma2_bf16(acc[b][0], acc[b][1], q.y, xq.y);
            fma2_bf16(acc[b][0], acc[b][1], q.z, xq.z);
            fma2_bf16(acc[b][0], acc[b][1], q.w, xq.w);
          }
        } else {
          const float wf[8] = {bf16_lo(q.x), bf16_hi(q.x), bf16_lo(q.y), bf16_hi(q.y),
                               bf16_lo(q.z), bf16_hi(q.z), bf16_lo(q.w), bf16_hi(q.w)};
#pragma unroll
          for (int b = 0; b < NB; ++b) {
            const uint4 xq = reinterpret_cast<const uint4*>(vec + static_cast<size_t>(b) * vec_elems)[J];
            const uint32_t xu[4] = {xq.x, xq.y, xq.z, xq.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              acc[b][0] = __fmaf_rn(wf[2 * u], bf16_lo(xu[u]), acc[b][0]);
              acc[b][1] = __fmaf_rn(wf[2 * u + 1], bf16_hi(xu[u]), acc[b][1]);
            }
          }
        }
      } else {
        const int slot0 = (J >> 5) * 64 + (J & 31);  // LayoutFp8 slots of vector J
        const uint32_t qu[4] = {q.x, q.y, q.z, q.w};
        if constexpr (kMixed) {
          uint32_t wp[8];
#pragma unroll
          for (int u = 0; u < 4; ++u) e4m3x4_to_bf16x2x2(qu[u], wp[2 * u], wp[2 * u + 1]);
#pragma unroll
          for (int b = 0; b < NB; ++b) {
            const uint4* xb = reinterpret_cast<const uint4*>(vec + static_cast<size_t>(b) * vec_elems);
            const uint4 x0 = xb[slot0], x1 = xb[slot0 + 32];
            const uint32_t xu[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
            for (int u = 0; u < 8; ++u) fma2_bf16(acc[b][0], acc[b][1], wp[u], xu[u]);
          }
        } else {
          float wf[16];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            wf[4 * u + 0] = e4m3_byte_scaled<0>(qu[u]);
            wf[4 * u + 1] = e4m3_byte_scaled<1>(qu[u]);
            wf[4 * u + 2] = e4m3_byte_scaled<2>(qu[u]);
            wf[4 * u + 3] = e4m3_byte_scaled<3>(qu[u]);
          }
#pragma unroll
          for (int b = 0; b < NB; ++b) {
            const uint4* xb = reinterpret_cast<const uint4*>(vec + static_cast<size_t>(b) * vec_elems);
            const uint4 x0 = xb[slot0], x1 = xb[slot0 + 32];
            const uint32_t xu[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              acc[b][0] = __fmaf_rn(wf[2 * u], bf16_lo(xu[u]), acc[b][0]);
              acc[b][1] = __fmaf_rn(wf[2 * u + 1], bf16_hi(xu[u]), acc[b][1]);
            }
          }
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
        float v = __fadd_rn(acc[b][0], acc[b][1]);
#pragma unroll
        for (int m = 16; m > 0; m >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, m));
        if constexpr (WT == MTP_W_FP8_E4M3) v = __fmul_rn(__fmul_rn(v, kE4m3Unscale), row_scale);
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
  argmax_finish<NB>(best, NB, wbest, a.ws, a.draft);
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
  ArgBest* wbest = reinterpret_cast<ArgBest*>(red + 2 * kWarps + 2);

  pdl_wait_prior_grid();
  for (int b = 0; b < nb; ++b) {
    rms_norm_to_smem<kThreads>(a.x + static_cast<size_t>(b) * H, a.final_norm_w, H, a.eps,
                               vec + static_cast<size_t>(b) * vec_elems, red, true, LayoutIdentity{});
    __syncthreads();
  }
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
  argmax_finish<kMaxB>(best, nb, wbest, a.ws, a.draft);
}

cudaError_t launch_sweep_kernel(void (*kernel)(SweepArgs), unsigned grid, size_t smem,
                                cudaStream_t stream, SweepArgs a) {
  void* args[] = {&a};
  return launch_pdl(reinterpret_cast<const void*>(kernel), dim3(grid), dim3(kThreads), smem, stream, args);
}

template <int WT, int NB>
cudaError_t launch_tma(SweepArgs a, const DeviceInfo& di, int64_t grid, size_t fixed,
                       cudaStream_t stream) {
  const size_t per_stage = static_cast<size_t>(kWarps) * (kChunk + 8);
  int S = static_cast<int>((static_cast<size_t>(di.smem_optin) - fixed) / per_stage);
  if (S > kMaxStages) S = kMaxStages;
  a.stages = S;
  const size_t smem = fixed + static_cast<size_t>(S) * per_stage;
  return launch_sweep_kernel(sweep_tma_kernel<WT, NB, MTP_MIXED_FMA != 0>, static_cast<unsigned>(grid),
                             smem, stream, a);
}

}  // namespace

size_t sweep_workspace_bytes(int B) {
  return static_cast<size_t>(kWsHeader) + static_cast<size_t>(kMaxGrid) * B * sizeof(ArgBest);
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
  int64_t grid = di.sm_count < want ? di.sm_count : want;
  if (grid > kMaxGrid) grid = kMaxGrid;
  if (grid < 1) grid = 1;
  const size_t misc = static_cast<size_t>(2 * kWarps + 2) * sizeof(float) +
                      static_cast<size_t>(kWarps) * kMaxB * sizeof(ArgBest) + 256;
  if (rows16 && a.B <= kTmaMaxB) {
    const int vec_elems = ((a.H / EPV + 31) / 32) * 32 * EPV;
    const size_t fixed = static_cast<size_t>(a.B) * vec_elems * 2 + misc;
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
  const size_t smem = static_cast<size_t>(a.B) * vec_elems * 2 + misc;
  if (smem > static_cast<size_t>(di.smem_optin)) return cudaErrorNotSupported;
  a.stages = 0;
  if (a.w_dtype == MTP_W_BF16)
    return launch_sweep_kernel(sweep_plain_kernel<MTP_W_BF16>, static_cast<unsigned>(grid), smem, stream, a);
  return launch_sweep_kernel(sweep_plain_kernel<MTP_W_FP8_E4M3>, static_cast<unsigned>(grid), smem, stream, a);
}

}  // namespace mtp
