// Input stage of the MTP draft head, one fused kernel ("glm5next_mtp_head.rs", `forward_one`:
// the embedding row read by pointer at token*hidden, `norm` with enorm into concat[0:H] and
// with hnorm into concat[H:2H], then the `eh_proj` dense gemv, n = H, k = 2H).
//
// Design: the same persistent, per-warp bulk-copy row stream as the output stage, here over the
// [H, 2H] eh_proj rows. The gather is an address computation on the device-resident token (so
// a draft chain or a CUDA graph can feed the previous draft straight back in), and every CTA
// builds the normalised concat of its B sequences in shared memory (one pass, one block
// reduction for all 2B norms) while its first weight stages are already in flight.
//
// Accuracy: the source's eh_proj gemv accumulates in FP32, and so does this kernel. Every
// product of two BF16 values is exact in fp32 (mixed-precision FMA); each lane keeps eight FP32
// accumulators per sequence (element e of a 16-byte vector goes to accumulator e), so an
// accumulator sums n = ceil(H / 128) exact products one FP32 rounding at a time. The 8 x 32
// accumulator values of a row are then added error-free (double-float TwoSum) and rounded once
// to BF16. x is therefore the BF16 rounding of a value within (n - 1) * 2^-24 * sum_k |w_k c_k|
// (first order) of the exact sum: at H = 6144, n = 48 and the band is below 2^-18.4 of the sum
// of |products|. An error-free sum of every product (TwoSum per product) had cost 7 us of a 30 us
// launch at the GLM size: the kernel is issue-bound there, not HBM-bound.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

namespace mtp {

namespace {

// Stage size and warps of the bulk-copy input kernel: 12 warps streaming 8 KB chunks (two in
// flight each) beat 16 warps with 4 KB chunks (30.6 vs 32.3 us at GLM size).
#ifndef MTP_IN_CHUNK
#define MTP_IN_CHUNK 8192
#endif
#ifndef MTP_INPUT_WARPS
#define MTP_INPUT_WARPS 12
#endif
constexpr int kInChunk = MTP_IN_CHUNK;
constexpr int kInWarps = MTP_INPUT_WARPS;
// Chunks at the start of each warp's run of eh_proj asked into L2 before the wait for the
// preceding kernel. In a draft chain that kernel is the sweep, whose last CTAs and grid argmax
// leave HBM partly idle, and so does this kernel's prologue (token, embedding row, the norms).
// Measured at H = 6144 (one GB300, 50-step chains): 2, 3, 5 and all (~10) chunks of 8 KB per
// warp took the BF16 step from 285 us to 283.1, 282.3, 281.5 and 281.6 us, the FP8 step from
// 166 us to 165.1, 164.3, 162.4 and 163.9 us. Real copies into the ring issued this early had
// cost 1.2 us a step instead: they hold shared memory and delay the prologue's own reads.
constexpr int kInL2Ahead = 5;

__device__ __forceinline__ bool token_ok(int32_t tok, int V) { return tok >= 0 && tok < V; }

// Build c_b = [enorm(embed[tok_b]) | hnorm(hidden_b)] for sequences b0 .. b0+nb-1 into shared
// memory (slot b - b0); valid[slot] says whether the token was in range.
template <int NT, class AfterLoads = NoOp>
__device__ void build_concat(const InputArgs& a, int b0, int nb, uint16_t* vec, int vec_elems,
                             float* red, bool* valid, AfterLoads after_loads = AfterLoads{}) {
  const int H = a.H;
  if (threadIdx.x < nb) {
    const bool ok = token_ok(a.tokens[b0 + threadIdx.x], a.V);
    valid[threadIdx.x] = ok;
    if (!ok) store_status(a.status, MTP_ERR_TOKEN_RANGE);
  }
  __syncthreads();
  auto job = [&](int j) {
    const int i = j >> 1, b = b0 + i;
    uint16_t* cb = vec + static_cast<size_t>(i) * vec_elems;
    if ((j & 1) == 0) {
      const bool ok = valid[i];
      const uint16_t* erow = ok ? a.embed + static_cast<int64_t>(a.tokens[b]) * H : a.embed;
      return NormJob{erow, a.enorm_w, cb, ok};
    }
    return NormJob{a.hidden + static_cast<size_t>(b) * H, a.hnorm_w, cb + H, true};
  };
  rms_norm_multi_to_smem<NT>(2 * nb, H, a.inv_h, a.eps, red, job, LayoutIdentity{}, after_loads);
  __syncthreads();
}

// One 16-byte weight vector (4 BF16 pairs) times the matching concat vector: element 2u goes to
// acc[2u], element 2u + 1 to acc[2u + 1], each an FMA with the exact product and one fp32
// rounding (mixed BF16 x BF16 -> FP32), eight independent chains.
__device__ __forceinline__ void dot8_fp32(const uint4& w, const uint4& c, float (&acc)[8]) {
  const uint32_t wu[4] = {w.x, w.y, w.z, w.w};
  const uint32_t cu[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int u = 0; u < 4; ++u) {
#if MTP_MIXED_FMA
    asm("{\n\t.reg .b16 wl, wh, cl, ch;\n\t"
        "mov.b32 {wl, wh}, %2;\n\tmov.b32 {cl, ch}, %3;\n\t"
        "fma.rn.f32.bf16 %0, wl, cl, %0;\n\tfma.rn.f32.bf16 %1, wh, ch, %1;\n\t}"
        : "+f"(acc[2 * u]), "+f"(acc[2 * u + 1])
        : "r"(wu[u]), "r"(cu[u]));
#else
    acc[2 * u] = __fmaf_rn(bf16_lo(wu[u]), bf16_lo(cu[u]), acc[2 * u]);
    acc[2 * u + 1] = __fmaf_rn(bf16_hi(wu[u]), bf16_hi(cu[u]), acc[2 * u + 1]);
#endif
  }
}

template <int NB, int NWI>
__global__ void __launch_bounds__(NWI * 32, 1) input_tma_kernel(const InputArgs a) {
  constexpr int NW = NWI;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ bool valid_s[kMaxB];

  const int S = a.stages;
  const int H = a.H;
  const int K = 2 * H;
  const int64_t row_bytes = static_cast<int64_t>(K) * 2;
  const int cpr = static_cast<int>((row_bytes + kInChunk - 1) / kInChunk);
  const uint32_t last_bytes = static_cast<uint32_t>(row_bytes - static_cast<int64_t>(cpr - 1) * kInChunk);
  const int vec_elems = ((K / 8 + 31) / 32) * 32 * 8;

  uint8_t* stages = smem;
  uint16_t* vec = reinterpret_cast<uint16_t*>(stages + static_cast<size_t>(NW) * S * kInChunk);
  uint64_t* bars = reinterpret_cast<uint64_t*>(vec + static_cast<size_t>(NB) * vec_elems);
  float* red = reinterpret_cast<float*>(bars + NW * S);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t r0 = static_cast<int64_t>(H) * blockIdx.x / gridDim.x;
  const int64_t r1 = static_cast<int64_t>(H) * (blockIdx.x + 1) / gridDim.x;
  const int cta_rows = static_cast<int>(r1 - r0);
  // The CTA's work is cta_rows x cpr chunks of 4 KB (row-major, i.e. contiguous in memory).
  // Warps take contiguous runs of equal length, so a row may be split between two warps (each
  // run is at least a row long, so never among more). Whole rows per warp left 2 or 3 rows
  // each at GLM size: the 3-row warps set the end. With fewer chunks than a row per warp the
  // runs stay row-aligned.
  const int F = cta_rows * cpr;
  const bool by_chunk = F / NW >= cpr;
  auto run_start = [&](int w) {
    return by_chunk ? static_cast<int>(static_cast<int64_t>(F) * w / NW)
                    : cpr * static_cast<int>(static_cast<int64_t>(cta_rows) * w / NW);
  };
  const int f0 = run_start(warp), f1 = run_start(warp + 1);
  const int nitems = f1 - f0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NW * S; ++i) mbar_init(smem_addr(&bars[i]), 1);
    fence_barrier_init();
  }
  __syncthreads();

  uint8_t* my_stages = stages + static_cast<size_t>(warp) * S * kInChunk;
  uint64_t* my_bars = bars + warp * S;
  const uint64_t policy = l2_evict_first_policy();
  const uint8_t* W = reinterpret_cast<const uint8_t*>(a.eh_proj);
  int pf = f0, ps = 0;
  auto issue_next = [&]() {
    const int64_t row = r0 + pf / cpr;
    const int pc = pf % cpr;
    const uint32_t bytes = (pc == cpr - 1) ? last_bytes : static_cast<uint32_t>(kInChunk);
    const uint8_t* src = W + row * row_bytes + static_cast<int64_t>(pc) * kInChunk;
    const uint32_t bar = smem_addr(&my_bars[ps]);
    mbar_arrive_expect_tx(bar, bytes);
    bulk_copy_g2s(smem_addr(my_stages + static_cast<size_t>(ps) * kInChunk), src, bytes, bar, policy);
    ++pf;
    if (++ps == S) ps = 0;
  };
  const int prefill = nitems < S ? nitems : S;
  // The weight stages are issued once the prologue has read the embedding row and
  // target_hidden: issued first, the weight stages of all SMs (~30 MB) sat in front of those
  // reads in the memory queues and delayed the prologue by several us.

  if (lane == 0 && nitems > 0) {
    // eh_proj does not depend on the preceding kernel; a warp's run is contiguous in memory
    auto off = [&](int f) { return static_cast<int64_t>(f / cpr) * row_bytes + static_cast<int64_t>(f % cpr) * kInChunk; };
    const int fe = (f0 + kInL2Ahead) < f1 ? (f0 + kInL2Ahead) : f1;
    const uint8_t* p0 = W + r0 * row_bytes + off(f0);
    const int64_t n = off(fe) - off(f0);
    if (((reinterpret_cast<uintptr_t>(p0) | static_cast<uintptr_t>(n)) & 15) == 0)
      bulk_prefetch_l2(p0, static_cast<uint32_t>(n));
  }
  // tokens and target_hidden may come from the preceding kernel
  pdl_wait_prior_grid();
  auto start_weights = [&]() {
    if (lane == 0)
      for (int t = 0; t < prefill; ++t) issue_next();
  };
  build_concat<NW * 32>(a, 0, NB, vec, vec_elems, red, valid_s, start_weights);
  bool valid[NB];
#pragma unroll
  for (int b = 0; b < NB; ++b) valid[b] = valid_s[b];
  pdl_launch_dependents();

  // partial sums of rows split between two warps: [warp][first | last][sequence]
  DF* part = reinterpret_cast<DF*>(red);
  float acc[NB][8];
#pragma unroll
  for (int b = 0; b < NB; ++b)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[b][e] = 0.0f;
  int cs = 0, t_fail = -1;
  uint32_t parity = 0;
  // the row's 8 x 32 accumulator values, added as double-floats (relative error ~2^-44)
  auto row_total = [&](int b) {
    DF v = df_add(df_add(df_add(DF{acc[b][0], 0.0f}, DF{acc[b][1], 0.0f}), df_add(DF{acc[b][2], 0.0f}, DF{acc[b][3], 0.0f})),
                  df_add(df_add(DF{acc[b][4], 0.0f}, DF{acc[b][5], 0.0f}), df_add(DF{acc[b][6], 0.0f}, DF{acc[b][7], 0.0f})));
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) v = df_add(v, shfl_xor_df(v, m));
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[b][e] = 0.0f;
    return v;
  };
  for (int t = 0; t < nitems; ++t) {
    const uint32_t bar = smem_addr(&my_bars[cs]);
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(bar, parity, a.wait_ns))) {
      t_fail = t;
      break;
    }
    const int f = f0 + t;
    const int cc = f % cpr;
    const uint4* wv = reinterpret_cast<const uint4*>(my_stages + static_cast<size_t>(cs) * kInChunk);
    const int nv = static_cast<int>(((cc == cpr - 1) ? last_bytes : static_cast<uint32_t>(kInChunk)) >> 4);
    const int J0 = cc * (kInChunk / 16);
#pragma unroll 2
    for (int j = lane; j < nv; j += 32) {
      const uint4 q = wv[j];
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        const uint4 cq = reinterpret_cast<const uint4*>(vec + static_cast<size_t>(b) * vec_elems)[J0 + j];
        dot8_fp32(q, cq, acc[b]);
      }
    }
    __syncwarp();
    if (lane == 0 && t + S < nitems) {
      fence_proxy_async_smem();
      issue_next();
    }
    if (++cs == S) { cs = 0; parity ^= 1u; }
    if (cc == cpr - 1 || t == nitems - 1) {
      // end of a row, or of this warp's run in the middle of one
      const int rl = f / cpr;
      const bool whole = rl * cpr >= f0 && cc == cpr - 1;
      const int slot = (cc == cpr - 1) ? 0 : 1;  // row finished here: its start was the previous warp's
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        const DF v = row_total(b);
        if (lane == 0) {
          if (whole) a.x[static_cast<size_t>(b) * H + r0 + rl] = valid[b] ? bf16_rne_df(v.hi, v.lo) : uint16_t(0);
          else part[(warp * 2 + slot) * NB + b] = v;
        }
      }
    }
  }
  if (t_fail >= 0 && lane == 0) {
    store_status(a.status, MTP_ERR_TIMEOUT);
    // let the copies still in flight land before the CTA's shared memory is released
    int s2 = cs;
    uint32_t par = parity;
    for (int u = t_fail; u < nitems && u < t_fail + S; ++u) {
      (void)mbar_wait_bounded(smem_addr(&my_bars[s2]), par);
      if (++s2 == S) { s2 = 0; par ^= 1u; }
    }
  }
  if (by_chunk) {
    // rows split at a warp boundary: the earlier warp's part (its "last") plus the later one's
    // ("first"), in that order
    __syncthreads();
    if (t_fail < 0 && threadIdx.x >= 1 && threadIdx.x < NW) {
      const int w = threadIdx.x, fb = run_start(w);
      if (fb % cpr != 0) {
        const int rl = fb / cpr;
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          const DF v = df_add(part[((w - 1) * 2 + 1) * NB + b], part[(w * 2 + 0) * NB + b]);
          a.x[static_cast<size_t>(b) * H + r0 + rl] = valid_s[b] ? bf16_rne_df(v.hi, v.lo) : uint16_t(0);
        }
      }
    }
  }
}

// Plain-load input stage for any H and B <= 16: one warp per output row. The concat of
// `group` sequences is resident at a time; larger batches take several passes over eh_proj.
__global__ void __launch_bounds__(kThreads) input_plain_kernel(const InputArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ bool valid_s[kMaxB];
  const int H = a.H, K = 2 * H, group = a.group;
  const int vec_elems = ((K + 7) / 8) * 8;
  uint16_t* vec = reinterpret_cast<uint16_t*>(smem);
  float* red = reinterpret_cast<float*>(vec + static_cast<size_t>(group) * vec_elems);

  pdl_wait_prior_grid();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
  const int64_t tw = static_cast<int64_t>(gridDim.x) * kWarps;
  for (int b0 = 0; b0 < a.B; b0 += group) {
    const int nb = (a.B - b0) < group ? (a.B - b0) : group;
    __syncthreads();  // the previous group's concat is no longer read
    build_concat<kThreads>(a, b0, nb, vec, vec_elems, red, valid_s);
    for (int64_t row = gw; row < H; row += tw) {
      const uint16_t* wr = a.eh_proj + row * K;
      for (int i = 0; i < nb; ++i) {
        const uint16_t* cb = vec + static_cast<size_t>(i) * vec_elems;
        DF acc{0.0f, 0.0f};
        for (int k = lane; k < K; k += 32)
          df_add(acc, __fmul_rn(bf16_bits_to_f32(wr[k]), bf16_bits_to_f32(cb[k])));
        for (int m = 16; m > 0; m >>= 1) acc = df_add(acc, shfl_xor_df(acc, m));
        if (lane == 0)
          a.x[static_cast<size_t>(b0 + i) * H + row] = valid_s[i] ? bf16_rne_df(acc.hi, acc.lo) : uint16_t(0);
      }
    }
  }
  pdl_launch_dependents();
}

cudaError_t launch_input_kernel(void (*kernel)(InputArgs), unsigned grid, unsigned threads, size_t smem,
                                cudaStream_t stream, InputArgs a) {
  void* args[] = {&a};
  return launch_pdl(reinterpret_cast<const void*>(kernel), dim3(grid), dim3(threads), smem, stream, args);
}

}  // namespace

cudaError_t launch_input_stage(const InputArgs& in, cudaStream_t stream) {
  DeviceInfo di;
  cudaError_t err = device_info(&di);
  if (err != cudaSuccess) return err;
  InputArgs a = in;
  const int K = 2 * a.H;
  const size_t misc = kRedBytes + 256;
  const bool rows16 = (K % 8) == 0;
  if (a.B >= MTP_TC_MIN_B) {
    bool launched = false;
    err = launch_input_tc(a, stream, &launched);
    if (launched || err != cudaSuccess) return err;
  }
  if (rows16 && a.B <= kTmaMaxB) {
    // the widest warp count whose stages fit next to the concat of B sequences
    const int vec_elems = ((K / 8 + 31) / 32) * 32 * 8;
    const size_t fixed = static_cast<size_t>(a.B) * vec_elems * 2 + misc;
    for (int nwi : {kInWarps, kWarps}) {
      const size_t per_stage = static_cast<size_t>(nwi) * (kInChunk + 8);
      if (fixed + 2 * per_stage > static_cast<size_t>(di.smem_optin)) continue;
      const int64_t want = (static_cast<int64_t>(a.H) + nwi - 1) / nwi;
      int64_t grid = di.sm_count < want ? di.sm_count : want;
      if (grid < 1) grid = 1;
      int S = static_cast<int>((static_cast<size_t>(di.smem_optin) - fixed) / per_stage);
      if (S > kMaxStages) S = kMaxStages;
      a.stages = S;
      const size_t smem = fixed + static_cast<size_t>(S) * per_stage;
      void (*k)(InputArgs) = nullptr;
      if (nwi == kInWarps) {
        switch (a.B) {
          case 1: k = input_tma_kernel<1, kInWarps>; break;
          case 2: k = input_tma_kernel<2, kInWarps>; break;
          case 3: k = input_tma_kernel<3, kInWarps>; break;
          default: k = input_tma_kernel<4, kInWarps>; break;
        }
      } else {
        switch (a.B) {
          case 1: k = input_tma_kernel<1, kWarps>; break;
          case 2: k = input_tma_kernel<2, kWarps>; break;
          case 3: k = input_tma_kernel<3, kWarps>; break;
          default: k = input_tma_kernel<4, kWarps>; break;
        }
      }
      return launch_input_kernel(k, static_cast<unsigned>(grid), nwi * 32, smem, stream, a);
    }
  }
  const int64_t want = (static_cast<int64_t>(a.H) + kWarps - 1) / kWarps;
  int64_t grid = di.sm_count < want ? di.sm_count : want;
  if (grid < 1) grid = 1;
  const int vec_elems = ((K + 7) / 8) * 8;
  const size_t per_seq = static_cast<size_t>(vec_elems) * 2;
  if (misc + per_seq > static_cast<size_t>(di.smem_optin)) return cudaErrorNotSupported;
  int group = static_cast<int>((static_cast<size_t>(di.smem_optin) - misc) / per_seq);
  if (group > a.B) group = a.B;
  a.stages = 0;
  a.group = group;
  const size_t smem = static_cast<size_t>(group) * per_seq + misc;
  return launch_input_kernel(input_plain_kernel, static_cast<unsigned>(grid), kThreads, smem, stream, a);
}

}  // namespace mtp
