// Batched output stage on the fifth-generation tensor cores: B = 2..16 sequences share one pass
// over lm_head ("glm5next_mtp_head.rs", `forward_one`: shared_head.norm, the lm_head gemv,
// argmax; here for a batch, as one skinny GEMM  logits[B, V] = xhat[B, H] . lm_head[V, H]^T
// fused with the argmax).
//
// The weights are the A operand straight from TMA (128-row tiles, 128-byte k-blocks, 128-byte
// swizzle: the K-major layout tcgen05.mma reads), the activations the B operand, the FP32
// accumulators in TMEM (32 columns per tile, 8 tiles at once). One thread issues the MMAs.
//  * BF16 head: kind::f16, xhat in BF16 (N = 16 sequence rows).
//  * FP8 head: kind::f8f6f4 with E4M3 on both sides, so the codes need no widening. xhat scaled
//    by a power of two per sequence (max |xhat| in [128, 256)) is split into two E4M3 values,
//    hi = e4m3(y) and lo = e4m3(16 (y - hi)): B has N = 32 rows, sequences 0..15 hi and 16..31 lo,
//    and a logit is (D_hi + D_lo / 16) 2^-k s_row. y has the 8 significant bits of a BF16 value
//    and hi keeps 4 of them, so y - hi is exact and has at most 4 bits left: lo holds it exactly
//    unless 16 (y - hi) falls below the E4M3 subnormal range (|xhat| below ~2^-11 of max |xhat|),
//    where the error stays under 2^-13 of max |xhat| per element.
// With every tile of a CTA in TMEM at once, each activation stage is built once per CTA (the
// mma.sync kernel rebuilds it for every group of 4 tiles, whose accumulators live in registers).
//
// Roles (192 threads):
//  * warps 0..3: the norm prologue, then builders of the activation stages (xhat rounded to
//    BF16 exactly as everywhere else), then the epilogue (warp w reads TMEM lanes 32w ..);
//  * warp 4 lane 0: TMA producer of the weight stages (6 x 32 KB ring);
//  * warp 5: TMEM allocation; lane 0 issues the MMAs.
// Every mbarrier wait is bounded; on a timeout the kernel records MTP_ERR_TIMEOUT and leaves
// after its own copies and MMAs are done.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "../../include/mtp_head.h"
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

#ifndef MTP_SWEEP_UMMA
#define MTP_SWEEP_UMMA 0  // 1: use this kernel for the batched sweep
#endif

namespace mtp {

namespace {

constexpr int kUThreads = 192;
constexpr int kUBuild = 128;          // warps 0..3
constexpr int kUProducerWarp = 4;
constexpr int kUMmaWarp = 5;
constexpr int kURows = 128;           // rows per tile (M)
constexpr int kUKS = 2;               // 128-byte k-blocks per stage
constexpr int kUATileBytes = kURows * 128;
constexpr int kUAStageBytes = kUKS * kUATileBytes;  // 32 KB
constexpr int kUAStages = 6;
constexpr int kUBStages = 3;
#ifndef MTP_UMMA_TILES
#define MTP_UMMA_TILES 8
#endif
constexpr int kUTiles = MTP_UMMA_TILES;  // tiles per group (32 TMEM columns each)
constexpr int kUCols = 32;
constexpr uint32_t kUTmemCols = kUTiles * kUCols <= 32 ? 32 : (kUTiles * kUCols <= 64 ? 64 : (kUTiles * kUCols <= 128 ? 128 : 256));
constexpr int kUSeq = 16;

template <int WT>
struct UCfg {
  static constexpr int kKbElems = (WT == MTP_W_BF16) ? 64 : 128;  // weights per 128-byte row segment
  static constexpr int kN = (WT == MTP_W_BF16) ? 16 : 32;         // B rows
  static constexpr int kBTileBytes = kN * 128;
  static constexpr int kBStageBytes = kUKS * kBTileBytes;
};

// Instruction descriptor, kind::f8f6f4: FP32 accumulator, E4M3 A and B (format 0), K-major.
__host__ __device__ constexpr uint32_t umma_idesc_e4m3(int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}
__device__ __forceinline__ void umma_e4m3(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Two fp32 values to E4M3 (round to nearest even, saturating): lo in bits 0..7, hi in 8..15.
__device__ __forceinline__ uint32_t e4m3x2_of(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
// The two E4M3 codes of the low 16 bits of w, as fp32 (exact).
__device__ __forceinline__ void e4m3x2_to_f32(uint32_t w, float& lo, float& hi) {
  asm("{\n\t.reg .b16 l, h0, h1;\n\t.reg .b32 p;\n\tmov.b32 {l, _}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 p, l;\n\tmov.b32 {h0, h1}, p;\n\tcvt.f32.f16 %0, h0;\n\tcvt.f32.f16 %1, h1;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(w));
}

__device__ void umma_argmax_finish(int nb, const ArgBest* wbest, uint8_t* ws, int32_t* draft) {
  __shared__ int is_last;
  ArgBest* part = reinterpret_cast<ArgBest*>(ws + kWsHeader);
  unsigned int* counter = reinterpret_cast<unsigned int*>(ws);
  if (threadIdx.x < nb) {
    ArgBest c{0.0f, -1};
    for (int w = 0; w < kUBuild / 32; ++w) {
      const ArgBest o = wbest[w * kUSeq + threadIdx.x];
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
    combine_partials(part, gridDim.x, nb, draft);
    if (threadIdx.x == 0) atomicExch(counter, 0u);
  }
}

template <int WT>
__global__ void __launch_bounds__(kUThreads, 1)
    sweep_umma_kernel(const __grid_constant__ CUtensorMap tmap_w, const SweepArgs a) {
  using Cfg = UCfg<WT>;
  constexpr int KBE = Cfg::kKbElems;
  constexpr int BTB = Cfg::kBTileBytes;
  constexpr int BSB = Cfg::kBStageBytes;
  constexpr bool kF8 = WT == MTP_W_FP8_E4M3;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint8_t* aring = smem;
  uint8_t* bring = aring + kUAStages * kUAStageBytes;
  uint64_t* afull = reinterpret_cast<uint64_t*>(bring + kUBStages * BSB);
  uint64_t* aempty = afull + kUAStages;
  uint64_t* bfull = aempty + kUAStages;
  uint64_t* bempty = bfull + kUBStages;
  uint64_t* dfull = bempty + kUBStages;   // a group's accumulators are final (MMA -> epilogue)
  uint64_t* dempty = dfull + 1;           // the epilogue has read them (epilogue -> MMA)
  uint64_t* mma_done = dempty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  float* nrm = reinterpret_cast<float*>(tmem_slot + 4);     // rh, rl, xs, us x kUSeq
  ArgBest* wbest = reinterpret_cast<ArgBest*>(nrm + 4 * kUSeq);
  DF* part = reinterpret_cast<DF*>(wbest + (kUBuild / 32) * kUSeq);
  float* mpart = reinterpret_cast<float*>(part + kUBuild / 32);
  DF* tot = reinterpret_cast<DF*>(mpart + kUBuild / 32);
  float* mtot = reinterpret_cast<float*>(tot + kUSeq);
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int B = a.B, H = a.H;
  const int64_t V = a.V;
  const int KB = (H + KBE - 1) / KBE;
  const int KP = (KB + kUKS - 1) / kUKS;
  const int T = static_cast<int>((V + kURows - 1) / kURows);
  const int t0 = static_cast<int>(static_cast<int64_t>(T) * blockIdx.x / gridDim.x);
  const int t1 = static_cast<int>(static_cast<int64_t>(T) * (blockIdx.x + 1) / gridDim.x);
  const int ngroups = (t1 - t0 + kUTiles - 1) / kUTiles;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kUAStages; ++i) {
      mbar_init(smem_addr(&afull[i]), 1);
      mbar_init(smem_addr(&aempty[i]), 1);
    }
    for (int i = 0; i < kUBStages; ++i) {
      mbar_init(smem_addr(&bfull[i]), kUBuild / 32);
      mbar_init(smem_addr(&bempty[i]), 1);
    }
    mbar_init(smem_addr(dfull), 1);
    mbar_init(smem_addr(dempty), kUBuild / 32);
    mbar_init(smem_addr(mma_done), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  for (int i = threadIdx.x; i < (kUBuild / 32) * kUSeq; i += kUThreads) wbest[i] = ArgBest{0.0f, -1};
  if (warp == kUMmaWarp) tmem_alloc(smem_addr(tmem_slot), kUTmemCols);
  tmem_fence_before_sync();
  __syncthreads();
  tmem_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == kUProducerWarp) {
    // ------------------------------------------------------------------ weight producer
    // The weights do not depend on the preceding kernels: the stream starts at once.
    if (lane == 0) {
      const uint64_t policy = l2_evict_first_policy();
      int slot = 0, issued = 0;
      uint32_t ep = 1;
      bool ok = true;
      for (int gi = 0; gi < ngroups && ok; ++gi) {
        const int g0 = t0 + gi * kUTiles;
        const int ntile = (t1 - g0) < kUTiles ? (t1 - g0) : kUTiles;
        for (int kp = 0; kp < KP && ok; ++kp) {
          const int nsub = KB - kp * kUKS < kUKS ? KB - kp * kUKS : kUKS;
          for (int j = 0; j < ntile; ++j) {
            if (*reinterpret_cast<volatile int*>(&abort_flag) || !mbar_wait_bounded(smem_addr(&aempty[slot]), ep)) {
              ok = false;
              break;
            }
            const uint32_t bar = smem_addr(&afull[slot]);
            mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nsub * kUATileBytes));
            for (int sb = 0; sb < nsub; ++sb)
              tma_load_2d(smem_addr(aring + slot * kUAStageBytes + sb * kUATileBytes), &tmap_w,
                          (kp * kUKS + sb) * KBE, (g0 + j) * kURows, bar, policy);
            ++issued;
            if (++slot == kUAStages) { slot = 0; ep ^= 1u; }
          }
        }
      }
      if (!ok) {
        store_status(a.status, MTP_ERR_TIMEOUT);
        atomicExch(&abort_flag, 1);
      }
      // every copy issued must land before the CTA's shared memory goes away
      for (int s = 0; s < kUAStages && s < issued; ++s) {
        const int uses = (issued - s + kUAStages - 1) / kUAStages;
        (void)mbar_wait_bounded(smem_addr(&afull[s]), static_cast<uint32_t>((uses - 1) & 1));
      }
    }
    __syncwarp();
  } else if (warp == kUMmaWarp) {
    // ------------------------------------------------------------------ MMA issue
    if (lane == 0) {
      constexpr uint32_t idesc = kF8 ? umma_idesc_e4m3(kURows, Cfg::kN) : umma_idesc_bf16(kURows, Cfg::kN);
      int aslot = 0, bslot = 0;
      uint32_t ap = 0, bp = 0;
      bool ok = true;
      for (int gi = 0; gi < ngroups && ok; ++gi) {
        const int g0 = t0 + gi * kUTiles;
        const int ntile = (t1 - g0) < kUTiles ? (t1 - g0) : kUTiles;
        // the accumulators are free once the epilogue has read the previous group
        if (gi > 0 && !mbar_wait_bounded(smem_addr(dempty), static_cast<uint32_t>((gi - 1) & 1))) {
          ok = false;
          break;
        }
        tmem_fence_after_sync();
        for (int kp = 0; kp < KP && ok; ++kp) {
          const int nsub = KB - kp * kUKS < kUKS ? KB - kp * kUKS : kUKS;
          if (*reinterpret_cast<volatile int*>(&abort_flag) || !mbar_wait_bounded(smem_addr(&bfull[bslot]), bp)) {
            ok = false;
            break;
          }
          const uint32_t bs = smem_addr(bring + bslot * BSB);
          for (int j = 0; j < ntile; ++j) {
            if (!mbar_wait_bounded(smem_addr(&afull[aslot]), ap)) {
              ok = false;
              break;
            }
            tmem_fence_after_sync();
            const uint32_t as = smem_addr(aring + aslot * kUAStageBytes);
            for (int sb = 0; sb < nsub; ++sb) {
              const uint64_t da = umma_desc_sw128(as + sb * kUATileBytes);
              const uint64_t db = umma_desc_sw128(bs + sb * BTB);
#pragma unroll
              for (int ks = 0; ks < 4; ++ks) {  // 32 bytes of k per MMA inside the 128-byte row
                const uint64_t koff = static_cast<uint64_t>((32 * ks) >> 4);
                const uint32_t acc = (kp | sb | ks) != 0 ? 1u : 0u;
                if constexpr (kF8)
                  umma_e4m3(tmem + static_cast<uint32_t>(j * kUCols), da + koff, db + koff, idesc, acc);
                else
                  umma_bf16(tmem + static_cast<uint32_t>(j * kUCols), da + koff, db + koff, idesc, acc);
              }
            }
            umma_commit(smem_addr(&aempty[aslot]));  // the weight stage is free once read
            if (++aslot == kUAStages) { aslot = 0; ap ^= 1u; }
          }
          umma_commit(smem_addr(&bempty[bslot]));  // the activation stage too, after every tile
          if (++bslot == kUBStages) { bslot = 0; bp ^= 1u; }
        }
        umma_commit(smem_addr(dfull));  // this group's accumulators are final
      }
      if (!ok) {
        store_status(a.status, MTP_ERR_TIMEOUT);
        atomicExch(&abort_flag, 1);
        umma_commit(smem_addr(dfull));  // wakes an epilogue waiting for this group
      }
      umma_commit(smem_addr(mma_done));
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ warps 0..3
    pdl_wait_prior_grid();  // x comes from the preceding kernel
    {
      auto row = [&](int b) -> const uint16_t* { return a.x + static_cast<size_t>(b) * H; };
      sumsq_rows<kUBuild, 8, kF8>(B, H, row, a.final_norm_w, part, mpart, tot, mtot, 1);
      if (threadIdx.x < kUSeq) {
        const int b = threadIdx.x;
        float rh = 0.0f, rl = 0.0f, xs = 1.0f, us = 1.0f;
        if (b < B) {
          // 1 / rms in fp64 (rsqrt: within an ulp or two of the correctly rounded value)
          const double ms = (static_cast<double>(tot[b].hi) + static_cast<double>(tot[b].lo)) * a.inv_h;
          const double rr = rsqrt(ms + static_cast<double>(a.eps));
          rh = static_cast<float>(rr);
          rl = static_cast<float>(rr - static_cast<double>(rh));
          if constexpr (kF8) {
            // largest |xhat| (rounding is monotonic, so it is the rounded max); scale it into
            // [128, 256)
            const float mx = mtot[b];
            const float yh = __fmul_rn(mx, rh);
            const float yl = __fmaf_rn(mx, rl, __fmaf_rn(mx, rh, -yh));
            const float m = bf16_bits_to_f32(bf16_rne_df(yh, yl));
            if (m > 0.0f && m <= 3.0e38f) {
              int e = 0;
              (void)frexpf(m, &e);
              xs = ldexpf(1.0f, 8 - e);
              us = ldexpf(1.0f, e - 8);
            }
          }
        }
        nrm[b] = rh;
        nrm[kUSeq + b] = rl;
        nrm[2 * kUSeq + b] = xs;
        nrm[3 * kUSeq + b] = us;
      }
      named_barrier_sync(1, kUBuild);
    }
    pdl_launch_dependents();

    int bslot = 0;
    uint32_t bep = 1;
    ArgBest best[kUSeq];
#pragma unroll
    for (int n = 0; n < kUSeq; ++n) best[n] = ArgBest{0.0f, -1};
    bool ok = true;
    for (int gi = 0; gi < ngroups && ok; ++gi) {
      const int g0 = t0 + gi * kUTiles;
      const int ntile = (t1 - g0) < kUTiles ? (t1 - g0) : kUTiles;
      // ---------------------------------------------------------------- builders
      // A stage holds kUKS k-blocks of B: k-block sb is Cfg::kN rows of 128 bytes, chunk c of row
      // n at swz(n, c). Cells: (sequence, k-block, chunk); BF16 8 activations, FP8 16 (hi and lo).
      constexpr int kCells = kUSeq * kUKS * 8;
      for (int kp = 0; kp < KP; ++kp) {
        if (*reinterpret_cast<volatile int*>(&abort_flag) ||
            !__all_sync(0xffffffffu, mbar_wait_bounded(smem_addr(&bempty[bslot]), bep))) {
          if (lane == 0) {
            store_status(a.status, MTP_ERR_TIMEOUT);
            atomicExch(&abort_flag, 1);
          }
          ok = false;
          break;
        }
        uint8_t* st = bring + bslot * BSB;
        for (int cell = threadIdx.x; cell < kCells; cell += kUBuild) {
          const int n = cell / (kUKS * 8), sb = (cell / 8) % kUKS, c = cell % 8;
          const int k0 = (kp * kUKS + sb) * KBE + (kF8 ? 16 : 8) * c;
          uint8_t* tile = st + sb * BTB;
          if constexpr (!kF8) {
            uint4 o = make_uint4(0u, 0u, 0u, 0u);
            if (n < B && k0 < H) {
              const uint4 xq = *reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(n) * H + k0);
              const uint4 wq = *reinterpret_cast<const uint4*>(a.final_norm_w + k0);
              const uint32_t xu[4] = {xq.x, xq.y, xq.z, xq.w};
              const float wf[8] = {bf16_lo(wq.x), bf16_hi(wq.x), bf16_lo(wq.y), bf16_hi(wq.y),
                                   bf16_lo(wq.z), bf16_hi(wq.z), bf16_lo(wq.w), bf16_hi(wq.w)};
              o = bf16x8_scaled_rne(xu, wf, nrm[n], nrm[kUSeq + n]);
            }
            *reinterpret_cast<uint4*>(tile + swz(n, c)) = o;
          } else {
            uint32_t hi[4] = {0u, 0u, 0u, 0u}, lo[4] = {0u, 0u, 0u, 0u};
            if (n < B && k0 < H) {
              const float xs = nrm[2 * kUSeq + n];
#pragma unroll
              for (int h = 0; h < 2; ++h) {  // two 8-element halves of the 16 codes
                const int kk = k0 + 8 * h;
                uint4 o = make_uint4(0u, 0u, 0u, 0u);
                if (kk < H) {
                  const uint4 xq = *reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(n) * H + kk);
                  const uint4 wq = *reinterpret_cast<const uint4*>(a.final_norm_w + kk);
                  const uint32_t xu[4] = {xq.x, xq.y, xq.z, xq.w};
                  const float wf[8] = {bf16_lo(wq.x), bf16_hi(wq.x), bf16_lo(wq.y), bf16_hi(wq.y),
                                       bf16_lo(wq.z), bf16_hi(wq.z), bf16_lo(wq.w), bf16_hi(wq.w)};
                  o = bf16x8_scaled_rne(xu, wf, nrm[n], nrm[kUSeq + n]);  // xhat, BF16
                }
                const uint32_t ou[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                  // y = xhat 2^k (exact); hi = e4m3(y); lo = e4m3(16 (y - hi)), y - hi exact
                  const float y0 = __fmul_rn(bf16_lo(ou[t]), xs), y1 = __fmul_rn(bf16_hi(ou[t]), xs);
                  const uint32_t hc = e4m3x2_of(y0, y1);
                  float h0, h1;
                  e4m3x2_to_f32(hc, h0, h1);
                  const uint32_t lc = e4m3x2_of(__fmul_rn(__fsub_rn(y0, h0), 16.0f), __fmul_rn(__fsub_rn(y1, h1), 16.0f));
                  const int q = 2 * h + (t >> 1);  // 32-bit word of the 16-byte chunk
                  hi[q] |= hc << (16 * (t & 1));
                  lo[q] |= lc << (16 * (t & 1));
                }
              }
            }
            *reinterpret_cast<uint4*>(tile + swz(n, c)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4*>(tile + swz(kUSeq + n, c)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
          }
        }
        fence_proxy_async_smem();  // generic stores, read by the tensor cores (async proxy)
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&bfull[bslot]));
        if (++bslot == kUBStages) { bslot = 0; bep ^= 1u; }
      }
      if (!ok) break;
      // ---------------------------------------------------------------- epilogue
      const bool done = mbar_wait_bounded(smem_addr(dfull), static_cast<uint32_t>(gi & 1));
      tmem_fence_after_sync();
      if (!done || *reinterpret_cast<volatile int*>(&abort_flag)) {
        if (!done && lane == 0) store_status(a.status, MTP_ERR_TIMEOUT);
        ok = false;
        break;
      }
      for (int j = 0; j < ntile; ++j) {
        uint32_t v[32];
        tmem_ld32(tmem + (static_cast<uint32_t>(32 * warp) << 16) + static_cast<uint32_t>(j * kUCols), v);
        const int64_t row = static_cast<int64_t>(g0 + j) * kURows + 32 * warp + lane;
        if (row < V) {
          const float rs = kF8 ? __ldg(a.scale + row) : 1.0f;
#pragma unroll
          for (int n = 0; n < kUSeq; ++n) {
            if (n < B) {
              float val = __uint_as_float(v[n]);
              if constexpr (kF8)
                val = __fmul_rn(__fmul_rn(__fmaf_rn(__uint_as_float(v[kUSeq + n]), 0.0625f, val), nrm[3 * kUSeq + n]), rs);
              if (a.logits != nullptr) a.logits[static_cast<int64_t>(n) * V + row] = val;
              arg_update(best[n], val, static_cast<int32_t>(row));
            }
          }
        }
      }
      tmem_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(dempty));
    }
    // per warp: the best of its 32 lanes for every sequence
#pragma unroll
    for (int n = 0; n < kUSeq; ++n) {
      ArgBest b = best[n];
#pragma unroll
      for (int m = 1; m < 32; m <<= 1) {
        const float v = __shfl_xor_sync(0xffffffffu, b.v, m);
        const int32_t i = __shfl_xor_sync(0xffffffffu, b.i, m);
        if (i >= 0) arg_update(b, v, i);
      }
      if (lane == 0 && n < B) wbest[warp * kUSeq + n] = b;
    }
  }
  tmem_fence_before_sync();
  __syncthreads();
  if (warp == kUMmaWarp) {
    // the accumulators are released only once every MMA issued into them is done
    if (lane == 0) (void)mbar_wait_bounded(smem_addr(mma_done), 0);
    __syncwarp();
    tmem_fence_after_sync();
    tmem_dealloc(tmem, kUTmemCols);
  }
  pdl_wait_prior_grid();  // the workspace may still be read by the kernel before (no-op if done)
  umma_argmax_finish(B, wbest, a.ws, a.draft);
}

template <int WT>
size_t umma_smem_bytes() {
  return 1024 + static_cast<size_t>(kUAStages) * kUAStageBytes + static_cast<size_t>(kUBStages) * UCfg<WT>::kBStageBytes +
         (2 * kUAStages + 2 * kUBStages + 3) * 8 + 16 + 4 * kUSeq * 4 + (kUBuild / 32) * kUSeq * sizeof(ArgBest) +
         (kUBuild / 32) * (sizeof(DF) + 4) + kUSeq * (sizeof(DF) + 4) + 64;
}

}  // namespace

cudaError_t launch_sweep_umma(const SweepArgs& a, cudaStream_t stream, bool* launched) {
  *launched = false;
  const int EB = (a.w_dtype == MTP_W_BF16) ? 2 : 1;
  if (!MTP_SWEEP_UMMA || a.B < 2 || a.B > kUSeq) return cudaSuccess;
  if ((static_cast<int64_t>(a.H) * EB) % 16 != 0 || (a.H % 16) != 0) return cudaSuccess;
  DeviceInfo di;
  cudaError_t err = device_info(&di);
  if (err != cudaSuccess) return err;
  const size_t smem = a.w_dtype == MTP_W_BF16 ? umma_smem_bytes<MTP_W_BF16>() : umma_smem_bytes<MTP_W_FP8_E4M3>();
  if (smem > static_cast<size_t>(di.smem_optin)) return cudaSuccess;
  const TmapEncodeFn enc = tensor_map_encoder();
  if (enc == nullptr) return cudaSuccess;
  CUtensorMap tm;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(a.H), static_cast<cuuint64_t>(a.V)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(a.H) * EB};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(a.w_dtype == MTP_W_BF16 ? 64 : 128), static_cast<cuuint32_t>(kURows)};
  const cuuint32_t estr[2] = {1, 1};
  if (enc(&tm, a.w_dtype == MTP_W_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
          const_cast<uint8_t*>(a.W), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaSuccess;
  const int64_t T = (static_cast<int64_t>(a.V) + kURows - 1) / kURows;
  int64_t g = di.sm_count < T ? di.sm_count : T;
  if (g > kMaxGrid) g = kMaxGrid;
  const unsigned grid = static_cast<unsigned>(g < 1 ? 1 : g);
  SweepArgs args = a;
  CUtensorMap tmc = tm;
  void* params[] = {&tmc, &args};
  *launched = true;
  const void* k = a.w_dtype == MTP_W_BF16 ? reinterpret_cast<const void*>(sweep_umma_kernel<MTP_W_BF16>)
                                          : reinterpret_cast<const void*>(sweep_umma_kernel<MTP_W_FP8_E4M3>);
  return launch_pdl(k, dim3(grid), dim3(kUThreads), smem, stream, params);
}

}  // namespace mtp
